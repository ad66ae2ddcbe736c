// Device helpers of the reducing kernels: streaming loads, bf16 unpacking,
// the packed (logit, id) key, per-lane top-k lists and warp reductions.
#pragma once

#include <cstdint>

#include "dvl_internal.h"

namespace dvl {

constexpr unsigned kFull = 0xffffffffu;

// 16-byte load of weights read exactly once: no L1 allocation, and ask L2
// to fetch the whole 256-byte span around the address.
__device__ __forceinline__ uint4 ld_stream16(const void *p)
{
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

// Programmatic dependent launch: allow the next kernel on the stream to
// start launching; wait until the preceding kernel has completed and its
// memory operations are visible.  Both are no-ops without a dependency.
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// The two bfloat16 halves of a 32-bit word as fp32 (exact: a bf16 is the
// upper half of a binary32).  The lower half is the element at the lower
// address.
__device__ __forceinline__ float bf16_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

// A candidate as one unsigned 64-bit key whose unsigned order is the result
// order: the upper word is the logit mapped to an order-preserving unsigned
// integer (-0 is folded onto +0; a NaN maps to 0, below every number), the
// lower word is 0xffffffff - full_id, so among equal logits the lower id has
// the larger key.  Key 0 marks an empty slot.
__device__ __forceinline__ uint64_t make_key(float logit, int32_t full_id)
{
    uint32_t b = __float_as_uint(logit);
    uint32_t mag = b & 0x7fffffffu;
    uint32_t hi;
    if (mag > 0x7f800000u)
        hi = 0u;                                  // NaN
    else if (mag == 0u)
        hi = 0x80000000u;                         // +0 and -0
    else
        hi = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
    return ((uint64_t)hi << 32) | (uint64_t)(0xffffffffu - (uint32_t)full_id);
}

__device__ __forceinline__ float key_logit(uint64_t key)
{
    uint32_t hi = (uint32_t)(key >> 32);
    uint32_t b = (hi & 0x80000000u) ? (hi & 0x7fffffffu) : ~hi;  // 0 -> NaN
    return __uint_as_float(b);
}

__device__ __forceinline__ int32_t key_id(uint64_t key)
{
    return (int32_t)(0xffffffffu - (uint32_t)key);  // empty slot -> -1
}

// A descending list of the KM best keys seen by one lane.
template <int KM>
struct TopList {
    uint64_t v[KM];
    __device__ __forceinline__ void init()
    {
#pragma unroll
        for (int i = 0; i < KM; ++i)
            v[i] = 0ull;
    }
    __device__ __forceinline__ void insert(uint64_t key)
    {
#pragma unroll
        for (int i = KM - 1; i > 0; --i)
            v[i] = key > v[i - 1] ? v[i - 1] : (key > v[i] ? key : v[i]);
        v[0] = key > v[0] ? key : v[0];
    }
    __device__ __forceinline__ void pop()
    {
#pragma unroll
        for (int i = 0; i + 1 < KM; ++i)
            v[i] = v[i + 1];
        v[KM - 1] = 0ull;
    }
};

__device__ __forceinline__ uint64_t warp_max_u64(uint64_t x)
{
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        uint64_t y = __shfl_xor_sync(kFull, x, off);
        x = y > x ? y : x;
    }
    return x;
}

// Take the warp's `k` best keys out of the lanes' lists, best first; every
// lane receives them.  Equal keys are taken one at a time (lowest lane first).
template <int KM>
__device__ __forceinline__ void warp_extract(TopList<KM> &L, int k, uint64_t (&out)[KM])
{
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int i = 0; i < KM; ++i) {
        out[i] = 0ull;
        if (i < k) {
            uint64_t head = L.v[0];
            uint64_t best = warp_max_u64(head);
            unsigned mask = __ballot_sync(kFull, head == best);
            if (lane == __ffs(mask) - 1)
                L.pop();
            out[i] = best;
        }
    }
}

__host__ __device__ constexpr int pow2_ceil(int x) { return x <= 1 ? 1 : 2 * pow2_ceil((x + 1) / 2); }
__host__ __device__ constexpr int log2_exact(int x) { return x <= 1 ? 0 : 1 + log2_exact(x / 2); }

// Reduce-scatter of P partial sums (P a power of two <= 32) across the warp:
// afterwards v[0] of lane l holds the warp-wide sum of value index
// (l >> (5 - log2 P)).  Each halving level sends half of the remaining
// values; once one value is left the remaining levels add it across lanes.
template <int P>
__device__ __forceinline__ void warp_reduce_scatter(float (&v)[P])
{
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int lvl = 0; lvl < 5; ++lvl) {
        const int off = 16 >> lvl;
        const int c = P >> lvl;  // values still held (compile-time after unrolling)
        if (c > 1) {
            const bool upper = (lane & off) != 0;
#pragma unroll
            for (int i = 0; i < c / 2; ++i) {
                float send = upper ? v[i] : v[i + c / 2];
                float keep = upper ? v[i + c / 2] : v[i];
                v[i] = keep + __shfl_xor_sync(kFull, send, off);
            }
        } else {
            v[0] += __shfl_xor_sync(kFull, v[0], off);
        }
    }
}

// Cross-block finish of a reducing kernel.  Every block calls it once, after
// its own candidates are final, with s_cand holding, for each of the M rows,
// `nlists` lists of KM keys ([M][nlists][KM] in shared memory; nlists is a
// multiple of 32, lane l of the merging warp takes lists l, l + 32, ...).
//  - k == 1: the block's best key per row goes to the workspace with a 64-bit
//    atomicMax; the last block to finish swaps each key back to 0 and writes
//    the id and the logit.
//  - k > 1: the block's k best keys per row go to its own workspace slots;
//    the last block merges every block's slots.
// The last block is found with a wrapping ticket (atomicInc up to
// gridDim.x - 1), so the ticket is 0 again when the call ends.  No block
// waits for another.
template <int KM>
__device__ __forceinline__ void block_finish(const uint64_t *s_cand, int M, int nlists,
                                             const ArgmaxArgs &a)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    unsigned int *ticket = reinterpret_cast<unsigned int *>(a.ws + kWsTicket);
    unsigned long long *best = reinterpret_cast<unsigned long long *>(a.ws + kWsBest);
    unsigned long long *slots = reinterpret_cast<unsigned long long *>(a.ws + kWsSlots);
    __shared__ int s_last;

    for (int m = warp; m < M; m += nwarps) {
        TopList<KM> L;
        L.init();
        for (int l = lane; l < nlists; l += 32)
#pragma unroll
            for (int i = 0; i < KM; ++i)
                L.insert(s_cand[(m * nlists + l) * KM + i]);
        if (KM == 1) {
            uint64_t key = warp_max_u64(L.v[0]);
            if (lane == 0 && key != 0ull)
                atomicMax(best + m, (unsigned long long)key);
        } else {
            uint64_t out[KM];
            warp_extract<KM>(L, a.k, out);
            // every lane holds out[]; lane i stores entry i
#pragma unroll
            for (int i = 0; i < KM; ++i)
                if (lane == i)
                    slots[((size_t)blockIdx.x * M + m) * KM + i] = out[i];
        }
    }
    __threadfence();  // this thread's slot stores before the ticket
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned int prev = atomicInc(ticket, gridDim.x - 1);
        s_last = (prev == gridDim.x - 1);
    }
    __syncthreads();
    if (!s_last)
        return;
    __threadfence();
    if constexpr (KM == 1) {
        // one thread per hidden row: the swaps go out together
        for (int m = threadIdx.x; m < M; m += blockDim.x) {
            uint64_t key = atomicExch(best + m, 0ull);
            a.ids[m] = key_id(key);
            a.logits[m] = key_logit(key);
        }
    } else {
        for (int m = warp; m < M; m += nwarps) {
            TopList<KM> L;
            L.init();
            for (int c = lane; c < (int)gridDim.x; c += 32)
#pragma unroll
                for (int i = 0; i < KM; ++i)
                    L.insert(__ldcg(slots + ((size_t)c * M + m) * KM + i));
            uint64_t out[KM];
            warp_extract<KM>(L, a.k, out);
            if (lane == 0) {
#pragma unroll
                for (int i = 0; i < KM; ++i)
                    if (i < a.k) {
                        a.ids[m * a.k + i] = key_id(out[i]);
                        a.logits[m * a.k + i] = key_logit(out[i]);
                    }
            }
        }
    }
}

}  // namespace dvl
