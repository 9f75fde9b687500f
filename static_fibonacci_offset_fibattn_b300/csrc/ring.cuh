// ring.cuh -- the persistent-CTA machinery shared by the tcgen05 attention kernels.
//
// A kernel runs min(tiles, 2 x SMs) CTAs; CTA b takes tiles b, b + grid, b + 2 grid, ...
// (consecutive tiles are consecutive 128-row blocks of one slice, so the CTAs in flight at
// any moment touch a narrow band of slices and their re-reads stay in L2).
//
// All shared-memory operands go through one in-order ring of slots (16 KB: 128 rows of 128
// bytes, or 17 KB where an item carries 8 extra rows after its tile): a producer warp
// walks the same per-tile item sequence as the consumers and fills slot (seq % slots) once
// the previous use of that slot has been released. A FULL barrier expects the producer's
// arrival with the TMA byte count (and, where a slot carries per-row side data copied by
// the producer's lanes, one more arrival per lane). Every EMPTY barrier expects one arrival
// per row warp of the kernel (`empty_arrivals`): that many tcgen05.commit's when the MMA warp
// consumed the slot, one arrival per row warp (lane 0 after __syncwarp) when the row warps
// did, or one arrival of that count for a staging slot.
#pragma once

#include <stdint.h>

#include "tc_prims.cuh"

namespace fibattn {
namespace ring {

constexpr uint32_t kSlotBytes = 16384;  // 128 rows x 128 bytes (64 bf16)

struct Tile {
    int32_t layer;   // launch layer
    int64_t zl;      // launch slice (layer * slices_per_layer + s)
    int32_t s;       // slice within the layer (b * heads + h)
    int32_t row0;    // first row of the tile in its slice
};

// idx < total tiles <= INT32_MAX (the launchers check), so 32-bit division suffices.
__device__ __forceinline__ Tile tile_of(uint32_t idx, uint32_t tiles_per_slice, uint32_t slices_per_layer) {
    Tile t;
    const uint32_t per_layer = tiles_per_slice * slices_per_layer;
    t.layer = (int32_t)(idx / per_layer);
    const uint32_t rem = idx - (uint32_t)t.layer * per_layer;
    const uint32_t s = rem / tiles_per_slice;
    t.zl = (int64_t)t.layer * slices_per_layer + s;
    t.s = (int32_t)s;
    t.row0 = (int32_t)(rem - s * tiles_per_slice) * 128;
    return t;
}

struct Ring {
    uint32_t base;            // shared address of slot 0 (1024-byte aligned)
    uint32_t full0;           // shared address of FULL[0]; EMPTY[i] follows the FULL array
    uint32_t slots;
    uint32_t empty_arrivals;  // = the kernel's number of row warps
    uint32_t slot_bytes = kSlotBytes;  // slot stride, a multiple of 1024

    __device__ __forceinline__ uint32_t slot(uint32_t seq) const { return seq % slots; }
    __device__ __forceinline__ uint32_t addr(uint32_t seq) const { return base + slot(seq) * slot_bytes; }
    __device__ __forceinline__ uint32_t full(uint32_t seq) const { return full0 + 8u * slot(seq); }
    __device__ __forceinline__ uint32_t empty(uint32_t seq) const { return full0 + 8u * (slots + slot(seq)); }
    __device__ __forceinline__ uint32_t parity(uint32_t seq) const { return (seq / slots) & 1u; }


    // producer: wait until the slot of `seq` is free
    __device__ __forceinline__ bool acquire(uint32_t seq, bool& aborted, int32_t* err) const {
        return tc::mbar_wait(empty(seq), parity(seq) ^ 1u, aborted, err);
    }
    // consumer: wait until the slot of `seq` holds its data. The parity wait is exact only if
    // the slot's previous use (seq - slots) is known to have landed (and, as always, `seq`
    // has not been released): a consumer that consumes every item of the ring in order meets
    // this by construction; one that skips other roles' items must know that by other means.
    __device__ __forceinline__ bool wait_full(uint32_t seq, bool& aborted, int32_t* err) const {
        return tc::mbar_wait(full(seq), parity(seq), aborted, err);
    }
    // row-warp release: every lane has finished reading the slot. The lanes read it with
    // generic loads and the next fill is a TMA write (the async proxy): without a proxy fence
    // the mbarrier hand-off orders only the generic proxy, and the refill may land in the slot
    // before those loads have read it.
    __device__ __forceinline__ void release_warp(uint32_t seq, int lane) const {
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(empty(seq));
    }
    // MMA-warp release: the slot is free once the MMAs issued so far have completed. All but
    // one of the EMPTY barrier's arrivals are made at once; the last is the commit, which
    // arrives when those MMAs complete, so the phase cannot complete before they do. (Each
    // tcgen05.commit costs the issuing thread about as much as an MMA; one per release keeps
    // them off the MMA warp's path.)
    __device__ __forceinline__ void release_mma(uint32_t seq) const {
        if (empty_arrivals > 1) tc::mbar_arrive_cnt(empty(seq), empty_arrivals - 1);
        tc::mma_commit(empty(seq));
    }
    // release of a staging slot by one thread, after its bulk store has read the slot
    __device__ __forceinline__ void release_stage(uint32_t seq) const {
        tc::mbar_arrive_cnt(empty(seq), empty_arrivals);
    }
    // producer side of a slot that is only staging space (no load): mark it owned
    __device__ __forceinline__ void publish_empty(uint32_t seq) const { tc::mbar_arrive(full(seq)); }
};

// Initialises FULL[slots] (full_arrivals each) and EMPTY[slots] (empty_arrivals each).
__device__ __forceinline__ void init_ring_barriers(const Ring& rg, uint32_t full_arrivals) {
    for (uint32_t i = 0; i < rg.slots; ++i) {
        tc::mbar_init(rg.full0 + 8u * i, full_arrivals);
        tc::mbar_init(rg.full0 + 8u * (rg.slots + i), rg.empty_arrivals);
    }
}

}  // namespace ring
}  // namespace fibattn
