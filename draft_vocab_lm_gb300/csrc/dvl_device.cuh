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

// Record a device-side failure in the workspace status word.
__device__ __forceinline__ void set_status(unsigned char *ws, unsigned int code)
{
    atomicOr(reinterpret_cast<unsigned int *>(ws + kWsStatus), code);
}

// Write result i (id and logit) of a call.  An id outside [0, V) -- a d2t
// entry out of range -- is written as it is and reported as
// DVL_ERR_OUT_OF_RANGE in the workspace status word.
__device__ __forceinline__ void put_result(const ArgmaxArgs &a, int i, uint64_t key)
{
    const int32_t id = key_id(key);
    if ((uint32_t)id >= (uint32_t)a.V)  // V <= 2^31 - 1; a negative id wraps high
        set_status(a.ws, 1u << DVL_ERR_OUT_OF_RANGE);
    a.ids[i] = id;
    a.logits[i] = key_logit(key);
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

// Insert key into a sorted (best first) list of KM keys in shared memory
// that only the calling thread uses; most keys lose to the last entry and
// cost one read.
template <int KM>
__device__ __forceinline__ void list_insert_smem(uint64_t *lst, uint64_t key)
{
    if (key <= lst[KM - 1])
        return;
    TopList<KM> t;
#pragma unroll
    for (int i = 0; i < KM; ++i)
        t.v[i] = lst[i];
    t.insert(key);
#pragma unroll
    for (int i = 0; i < KM; ++i)
        lst[i] = t.v[i];
}

// The cross-block ticket: a wrapping increment (atomicInc semantics) with
// release and acquire at GPU scope.  Release: the calling block's earlier
// writes (made before a __syncthreads, by any of its threads) are visible
// to whoever observes the increment; acquire: the caller's later reads (and,
// after a __syncthreads, its block's) see what every earlier incrementer
// released.  One round trip, where a full fence on each side costs far more
// while the next kernel's loads crowd the memory system.
__device__ __forceinline__ unsigned int ticket_inc(unsigned int *p, unsigned int lim)
{
    unsigned int old;
    asm volatile("atom.acq_rel.gpu.global.inc.u32 %0, [%1], %2;"
                 : "=r"(old)
                 : "l"(p), "r"(lim)
                 : "memory");
    return old;
}

__device__ __forceinline__ uint64_t warp_max_u64(uint64_t x)
{
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        uint64_t y = __shfl_xor_sync(kFull, x, off);
        x = y > x ? y : x;
    }
    return x;
}

// Butterfly merge of the lanes' lists: afterwards every lane's list holds
// the warp's KM best keys (KM a power of two), best first.  At each level a
// lane swaps lists with its partner; the elementwise maximum of one
// descending list and the other reversed holds the KM largest keys of both
// as a bitonic sequence, which a bitonic merge network puts in order.
// `width` (a power of two <= 32) limits the merge to aligned groups of that
// many lanes; each group ends with its own best keys.
template <int KM>
__device__ __forceinline__ void warp_merge_topk(TopList<KM> &L, int width = 32)
{
    static_assert((KM & (KM - 1)) == 0, "KM must be a power of two");
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        if (off >= width)
            continue;
        uint64_t o[KM];
#pragma unroll
        for (int i = 0; i < KM; ++i)
            o[i] = __shfl_xor_sync(kFull, L.v[i], off);
#pragma unroll
        for (int i = 0; i < KM; ++i) {
            const uint64_t b = o[KM - 1 - i];
            L.v[i] = b > L.v[i] ? b : L.v[i];
        }
#pragma unroll
        for (int st = KM / 2; st >= 1; st >>= 1)
#pragma unroll
            for (int i = 0; i < KM; ++i)
                if ((i & st) == 0) {
                    const uint64_t x = L.v[i], y = L.v[i + st];
                    L.v[i] = x > y ? x : y;
                    L.v[i + st] = x > y ? y : x;
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

// Merge, for every hidden row m < M, nl sorted lists of KM keys (list c of
// row m at src + (m * stride + c) * KM, read from L2) into the row's KM best
// keys, handed over as emit(m, i, key) for i < KM, best first.  Every thread
// of the block must call it (one of its two layouts meets at a
// __syncthreads).  A warp's lanes read consecutive lists 16 bytes at a
// time, kBatch lists each before inserting any (one L2 round trip per
// batch).
template <int KM, typename Emit>
__device__ __forceinline__ void merge_lists(const uint64_t *src, int stride, int nl, int M,
                                            Emit emit)
{
    static_assert(KM % 2 == 0, "lists are read in pairs of keys");
    constexpr int kBatch = 8;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    auto gather = [&](TopList<KM> &L, int m, int c_first, int c_step) {
        const uint64_t *row = src + (size_t)m * stride * KM;
        for (int c0 = c_first; c0 < nl; c0 += kBatch * c_step) {
            ulonglong2 v[kBatch][KM / 2];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int c = c0 + u * c_step;
#pragma unroll
                for (int i = 0; i < KM / 2; ++i)
                    v[u][i] = c < nl ? __ldcg(reinterpret_cast<const ulonglong2 *>(
                                           row + (size_t)c * KM) + i)
                                     : make_ulonglong2(0ull, 0ull);
            }
            // each list is sorted best first: once one of its keys loses to
            // the current k-th best, so does the rest
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                uint64_t key[KM];
#pragma unroll
                for (int i = 0; i < KM / 2; ++i) {
                    key[2 * i] = v[u][i].x;
                    key[2 * i + 1] = v[u][i].y;
                }
#pragma unroll
                for (int i = 0; i < KM; ++i) {
                    if (key[i] <= L.v[KM - 1])
                        break;
                    L.insert(key[i]);
                }
            }
        }
    };
    auto pick = [](const TopList<KM> &F, int i) {
        uint64_t key = F.v[0];
#pragma unroll
        for (int j = 1; j < KM; ++j)
            key = i == j ? F.v[j] : key;
        return key;
    };
    if (M >= nwarps) {
        // tpr threads per hidden row (a power of two, at most a warp), every
        // row in one pass, no block-wide step
        int tpr = 32;
        while (tpr * M > (int)blockDim.x)
            tpr >>= 1;
        const int m = threadIdx.x / tpr, sub = threadIdx.x % tpr;
        TopList<KM> L;
        L.init();
        if (m < M)
            gather(L, m, sub, tpr);
        warp_merge_topk<KM>(L, tpr);
        if (m < M && sub < KM)
            emit(m, sub, pick(L, sub));
    } else {
        // nwarps / M warps per hidden row, merged through shared memory
        constexpr int kFinWarps = 32;  // the most warps a block can have
        __shared__ uint64_t s_fin[kFinWarps][KM];
        const int wpm = nwarps / M;
        const int m = warp % M, q = warp / M;
        TopList<KM> L;
        L.init();
        if (q < wpm)
            gather(L, m, 32 * q + lane, 32 * wpm);
        warp_merge_topk<KM>(L);
        if (lane == 0) {
#pragma unroll
            for (int i = 0; i < KM; ++i)
                s_fin[warp][i] = q < wpm ? L.v[i] : 0ull;
        }
        __syncthreads();
        if (warp < M) {
            TopList<KM> F;  // the warps' lists are already in order
#pragma unroll
            for (int i = 0; i < KM; ++i)
                F.v[i] = lane < wpm ? s_fin[warp + M * lane][i] : 0ull;
            warp_merge_topk<KM>(F);
            if (lane < KM)
                emit(warp, lane, pick(F, lane));
        }
    }
}

// Cross-block finish of a reducing kernel.  Every block calls it once, after
// its own candidates are final, with s_cand holding, for each of the M rows,
// `nlists` lists of KM keys ([M][nlists][KM] in shared memory; lane l of
// the merging warp takes lists l, l + 32, ...).
//  - k == 1: the block's best key per row goes to the workspace with a 64-bit
//    atomicMax; the last block to finish swaps each key back to 0 and writes
//    the id and the logit.
//  - k > 1: the block's k best keys per row go to its own workspace slots
//    ([M][blocks][k]).  The last block merges every block's slots; or, when
//    that is many lists (M * blocks >= kTwoLevelLists, and more than kGroup
//    blocks), merging is two-level: the last block of each group of kGroup
//    blocks (by a group ticket) merges the group's slots into the group's
//    list, and the last of those (by the main ticket) merges the group lists
//    -- the final merge reads blocks / kGroup lists per row, not one per
//    block.  (Measured on the tcgen05 grid of 138 blocks: top-4 at 32 rows
//    3.5 us faster, at 20 rows 2 us; below the threshold the extra ticket
//    round trip costs more than it saves: +0.85 us at 8 rows on 304
//    blocks.)
// The last block (of a group, or of the grid) is found with a wrapping
// ticket (an increment up to its count - 1 that wraps), so every ticket is
// 0 again when the call ends.  No block waits for another.
template <int KM>
__device__ __forceinline__ void block_finish(const uint64_t *s_cand, int M, int nlists,
                                             const ArgmaxArgs &a)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    unsigned int *ticket = reinterpret_cast<unsigned int *>(a.ws + kWsTicket);
    unsigned long long *best = reinterpret_cast<unsigned long long *>(a.ws + kWsBest);
    uint64_t *slots = reinterpret_cast<uint64_t *>(a.ws + kWsSlots);
    // top-k: groups of kGroup blocks, their group lists and group tickets
    // after the slots (the slot area is sized for kMaxCtas blocks)
    const int G = (int)gridDim.x;
    const int ngrp = (KM == 1 || M * G < kTwoLevelLists) ? 1 : (G + kGroup - 1) / kGroup;
    uint64_t *gslots = slots + (size_t)kMaxCtas * M * KM;
    unsigned int *gtickets = reinterpret_cast<unsigned int *>(gslots + (size_t)kMaxGroups * M * KM);
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
            warp_merge_topk<KM>(L);
            // every lane holds the list; lane i stores entry i
#pragma unroll
            for (int i = 0; i < KM; ++i)
                if (lane == i)
                    slots[((size_t)m * gridDim.x + blockIdx.x) * KM + i] = L.v[i];
        }
    }
    __syncthreads();  // the block's keys and slots, then its ticket (release)
    if (threadIdx.x == 0) {
        if (ngrp == 1) {
            const unsigned int prev = ticket_inc(ticket, (unsigned int)G - 1u);
            s_last = (prev == (unsigned int)G - 1u);
        } else {
            // top-k on more than kGroup blocks: first the group's ticket
            const int g = (int)blockIdx.x / kGroup;
            const unsigned int gs = (unsigned int)min(kGroup, G - g * kGroup);
            const unsigned int prev = ticket_inc(gtickets + g, gs - 1u);
            s_last = (prev == gs - 1u);
        }
    }
    __syncthreads();  // the last block's reads follow its acquire
    if (!s_last)
        return;
    if constexpr (KM == 1) {
        // one thread per hidden row: the swaps go out together
        for (int m = threadIdx.x; m < M; m += blockDim.x) {
            put_result(a, m, atomicExch(best + m, 0ull));
        }
    } else {
        auto emit_out = [&](int m, int i, uint64_t key) {
            if (i < a.k)
                put_result(a, m * a.k + i, key);
        };
        if (ngrp == 1) {
            merge_lists<KM>(slots, G, G, M, emit_out);
            return;
        }
        // this block is its group's last: the group's lists -> its group list
        const int g = (int)blockIdx.x / kGroup;
        const int gs = min(kGroup, G - g * kGroup);
        merge_lists<KM>(slots + (size_t)g * kGroup * KM, G, gs, M,
                        [&](int m, int i, uint64_t key) {
                            gslots[((size_t)m * ngrp + g) * KM + i] = key;
                        });
        __syncthreads();  // the group list, then the top ticket (release)
        if (threadIdx.x == 0) {
            const unsigned int prev = ticket_inc(ticket, (unsigned int)ngrp - 1u);
            s_last = (prev == (unsigned int)ngrp - 1u);
        }
        __syncthreads();
        if (!s_last)
            return;
        merge_lists<KM>(gslots, ngrp, ngrp, M, emit_out);
    }
}

}  // namespace dvl
