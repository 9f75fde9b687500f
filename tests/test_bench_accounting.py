"""The benchmark's roofline accounting, without a GPU: the algorithmic bytes per query token
of each kernel equal the counts of rows that kernel must read and write once (q, k, v, o, dO,
lse and the gradients; bf16 rows of 128 B at head size 64), grouped-query workloads share their
k/v rows among the heads that read them, and every kernel the library times has an entry, so
the reported roofline fraction is never computed from a missing figure."""
import os
import re
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import fibattn_inputs as fi  # noqa: E402

CSRC = os.path.join(ROOT, "static_fibonacci_offset_fibattn_b300", "csrc")
ROW_BF16_64 = 64 * 2   # one row at head size 64, bf16
ROW_F32_64 = 64 * 4
LSE = 4


def _tokens(spec):
    return spec["Lc"] * spec["B"] * spec["H"] * spec["T"]


def test_forward_bytes_per_token():
    c5 = fi.WORKLOADS["c5"]
    # q, k, v read once, o written once, lse written once
    assert bench.algo_bytes("fwd_tc_bf16", c5) == 3 * ROW_BF16_64 + ROW_BF16_64 + LSE == 516
    # the fp32 single layer reads and writes fp32 rows
    assert bench.algo_bytes("fwd_simt_f32", fi.WORKLOADS["c1"]) == 4 * ROW_F32_64 + LSE == 1028
    # head size 128: rows twice as long
    assert bench.algo_bytes("fwd_tc128_bf16", fi.WORKLOADS["c5w"]) == 4 * 2 * ROW_BF16_64 + LSE


def test_backward_bytes_per_token_and_launch():
    c5 = fi.WORKLOADS["c5"]
    # query owner: q, k, v, o, dO and lse in, dq out
    assert bench.algo_bytes("bwd_dq_tc", c5) == 5 * ROW_BF16_64 + LSE + ROW_BF16_64 == 772
    # key owner: q, k, v, dO and lse in, dk and dv out
    assert bench.algo_bytes("bwd_dkdv_tc", c5) == 4 * ROW_BF16_64 + LSE + 2 * ROW_BF16_64 == 772
    # the figure the bench reports as the dominant kernel's bytes per launch at c5
    assert bench.algo_bytes("bwd_dkdv_tc", c5) * _tokens(c5) == 809_500_672


def test_grouped_query_heads_share_kv_rows():
    c5g = fi.WORKLOADS["c5g"]
    G = c5g["H"] // c5g["Hkv"]
    assert G > 1
    share = 1 - 1 / G
    # the forward reads k and v once per kv head: two of its rows shrink by (1 - 1/G)
    assert bench.algo_bytes("fwd_tc_bf16", c5g) == pytest.approx(516 - 2 * ROW_BF16_64 * share)
    # the key owner also writes dk, dv once per kv head: four rows shrink
    assert bench.algo_bytes("bwd_dkdv_tc", c5g) == pytest.approx(772 - 4 * ROW_BF16_64 * share)
    # a kernel without k/v-shaped rows is unchanged
    assert bench.algo_bytes("dalpha_reduce", c5g) == bench.ALGO_BYTES["dalpha_reduce"]


def _timed_kernel_names():
    """Kernel names the library registers for its per-kernel event timing (KernelScope)."""
    names = set()
    for f in os.listdir(CSRC):
        if f.endswith(".cu"):
            text = open(os.path.join(CSRC, f)).read()
            names |= set(re.findall(r'"((?:fwd|bwd|rope|dalpha)_[a-z0-9_]+)"', text))
    return names


def test_every_timed_kernel_has_an_accounting_entry():
    # the cos/sin table is built once per (T, base), outside any timed step
    setup_only = {"rope_table"}
    names = _timed_kernel_names() - setup_only
    assert names, "no kernel names found in the sources"
    missing = sorted(n for n in names if n not in bench.ALGO_BYTES)
    assert not missing, missing
    # and its committed ncu traffic figures are keyed to an existing source file
    for kernel, src in bench.KERNEL_SRC.items():
        assert os.path.exists(os.path.join(CSRC, src)), (kernel, src)
    assert set(bench.KERNEL_SRC) <= set(bench.ALGO_BYTES)


def test_kernel_roofline_record():
    # one launch covers at most 16 layers; achieved = algorithmic bytes per launch / mean time
    c5 = fi.WORKLOADS["c5"]
    per_kernel = {"bwd_dkdv_tc": (2 * 0.369, 2)}  # two launches of 369 us
    r = bench.kernel_roofline("bwd_dkdv_tc", per_kernel, c5, "c5", 6508.2, "measured")
    assert r["algorithmic_bytes_per_launch"] == 809_500_672
    assert r["avg_launch_us"] == pytest.approx(369.0)
    assert r["achieved"] == pytest.approx(809_500_672 / 369e-6 / 1e9, rel=1e-3)
    assert r["frac"] == pytest.approx(r["achieved"] / 6508.2, abs=1e-4)
    # a 32-layer call is two launches of 16 layers each: bytes per launch halve
    c5_32 = dict(c5, Lc=32)
    r32 = bench.kernel_roofline("bwd_dkdv_tc", per_kernel, c5_32, "c5", 6508.2, "measured")
    assert r32["algorithmic_bytes_per_launch"] == 809_500_672


def test_dense_context_flops():
    # causal attention over T keys: query i attends i + 1 keys, 4 d flops per (query, key)
    # (q.k and p.v), so 4 d T (T + 1) / 2 per (b, h) slice; at the 4x-length shape, B2 H8:
    c4 = fi.WORKLOADS["c4"]
    T, d = c4["T"], c4["d"]
    brute = sum(4 * d * (i + 1) for i in range(T)) * c4["B"] * c4["H"]
    assert brute == 4 * d * T * (T + 1) // 2 * c4["B"] * c4["H"]
    assert round(brute / 1e9, 2) == 34.37


def test_fused_rope_forward_is_accounted_like_the_forward():
    # the table rows it reads are L2-resident reuse, not compulsory traffic
    c3r = fi.WORKLOADS["c3r"]
    assert bench.algo_bytes("fwd_rope_tc_bf16", c3r) == bench.algo_bytes("fwd_tc_bf16", c3r) == 516
    assert c3r.get("rope_fused") and "rope_base" in c3r


def test_one_pass_backward_bytes_per_token():
    # the one-pass backward reads q, k, v, dO, D and lse log2(e) once and writes dq, dk, dv
    # once; its pre-pass reads o, dO and lse and writes D and lse log2(e): together they count
    # the D/lse round trip once more than the two-kernel query owner, which forms D itself
    c5o = fi.WORKLOADS["c5o"]
    assert bench.algo_bytes("bwd_fused_tc", c5o) == 4 * ROW_BF16_64 + 2 * 4 + 3 * ROW_BF16_64
    assert bench.algo_bytes("bwd_prep", c5o) == 2 * ROW_BF16_64 + LSE + 2 * 4
    assert bench.KERNEL_SRC["bwd_fused_tc"] == bench.KERNEL_SRC["bwd_prep"] == "bwd_fused.cu"
    c5 = fi.WORKLOADS["c5"]
    assert {k: v for k, v in c5o.items() if k not in ("desc", "bwd_fused")} == \
        {k: v for k, v in c5.items() if k != "desc"}


def test_committed_traffic_covers_the_current_sources():
    # the bench reports DRAM traffic from profiles/ncu_traffic.txt only for the kernel source
    # it was captured on (a sha256 prefix); the default run's kernels must have a line for
    # their current sources, else the roofline records carry traffic null
    for kernel, workload in [("fwd_tc_bf16", "c4"), ("fwd_tc_bf16", "c5"), ("bwd_dq_tc", "c5"),
                             ("bwd_dkdv_tc", "c5"), ("bwd_fused_tc", "c5o"), ("bwd_prep", "c5o")]:
        t = bench.committed_traffic(kernel, workload)
        assert t is not None, (kernel, workload, "recapture its traffic line on the current source")
        assert 100.0 < t < 2000.0, (kernel, workload, t)
