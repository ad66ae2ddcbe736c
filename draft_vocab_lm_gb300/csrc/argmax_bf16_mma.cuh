// Fused skinny projection + argmax / top-k over a bf16 draft head, on the
// register-path tensor cores, for the unrolled hidden widths (2,560 and
// 5,120), three to eight hidden rows and heads of at least one full 8-row
// tile per warp.  ("Shortlist MTP", sections "What I was
// testing" and "What was actually happening": a hidden row of width 2,560
// against every head row, M = 1 or 3 -- bandwidth-heavy, for a couple of
// rows; the skinny low-M kernel and the local argmax reduction.)
//
// Why tensor cores for a memory-bound product: on CUDA cores every 16 bytes
// of weights cost 8 widenings and 8 M fused multiply-adds, about 35 issued
// instructions at M = 3, and the issue slots, not HBM, set the pace.  Here
// every 32 bytes cost one load and four MMAs at any M <= 8 (and at 5 .. 8
// rows it streams faster than the tcgen05 kernel's 128-row tiles).  The
// price is that a row streams through 4 lanes instead of 32: a warp with a
// short range spends more memory round trips on it, so one or two hidden
// rows and heads of fewer rows stay on the CUDA cores.
//
// Operands of mma.sync m16n8k16 (bf16 in, fp32 accumulate):
//   - B (16 k x 8 n) is 8 head rows: lane (g, q) = (lane / 4, lane % 4)
//     supplies column n = g, i.e. head row g of the tile, straight from the
//     16-byte loads it issued (no conversion);
//   - A (16 m x 16 k) is the hidden rows: lane (g, q) supplies rows g and
//     g + 8 (rows 8..15 are zero when M <= 8); rows at or past M hold a copy
//     of a valid row, and only feed result rows that nobody reads;
//   - the k order inside an MMA is a permutation of the weights' k, the same
//     for A and B: the k slots 2q, 2q + 1, 2q + 8, 2q + 9 of lane (g, q) are
//     the weights kb .. kb + 3 with kb = 128 c + 64 w + 16 q + 4 s for chunk
//     c, load w < 2 and quarter s < 4 of the lane's 32-byte load, so every
//     product pairs the right weight and hidden value and every k is used
//     once;
//   - D lane (g, q) ends with the logits of hidden rows g and g + 8 against
//     head rows 2q and 2q + 1 of the tile.
//
// Work split as in the CUDA-core kernel: a persistent grid of two 256-thread
// blocks per SM, one balanced contiguous row range per warp, walked in tiles
// of 8 rows (the last one partial).  Lane (g, q) streams, per 128-wide k
// chunk, 32 bytes of row g at 32 q + 128 w bytes for w < 2 (one 256-bit
// load each), so each warp load instruction reads one whole 128-byte line of
// each of 8 rows.  The head must be 32-byte aligned.  NB chunks
// run ahead of the MMAs through a register ring, across tile boundaries; a
// head the caller marked static starts filling it before the wait for the
// preceding kernel.  The hidden rows are copied into shared memory as bf16
// (asynchronous 16-byte copies), each row padded by 16 bytes so that the
// lanes of one load phase hit distinct banks.  Results go through the same
// per-lane lists, block merge and cross-block finish as the other kernels.
#pragma once

#include <cuda_runtime.h>

#include "dvl_device.cuh"

namespace dvl {
namespace bf16mma {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kTile = 8;        // head rows per MMA tile (MMA n)
constexpr int kChunk = 128;     // weights per row per k chunk (2 loads per lane)
constexpr int kLists = kWarps * 4;  // per hidden row per block: lanes (g = m, q < 4) of each warp
constexpr int kAcc = 4;         // independent accumulators (MMA dependency chains)
constexpr int kMaxRows = 16;    // hidden rows per launch (rows of the A operand)

// D += A B for one m16n8k16 MMA: a0 / a2 hold A row g, a1 / a3 row g + 8.
__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 32-byte load of weights read exactly once (no L1 allocation, 256-byte L2
// fetch); lo holds the lower 16 bytes.
__device__ __forceinline__ void ld_stream32(const void *p, uint4 &lo, uint4 &hi)
{
    asm("ld.global.nc.L1::no_allocate.L2::256B.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
        : "=r"(lo.x), "=r"(lo.y), "=r"(lo.z), "=r"(lo.w), "=r"(hi.x), "=r"(hi.y), "=r"(hi.z),
          "=r"(hi.w)
        : "l"(p));
}

__device__ __forceinline__ void cp_async16(void *dst, const void *src)
{
    const unsigned d = (unsigned)__cvta_generic_to_shared(dst);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src) : "memory");
}

// Staged hidden row pitch in bf16 elements: K plus 8 (16 bytes).
template <int KC> __host__ __device__ constexpr int pitch() { return KC + 8; }

template <int M, int KM, int KC>
__host__ __device__ constexpr size_t smem_bytes()
{
    return (size_t)M * pitch<KC>() * 2 + (size_t)M * kLists * KM * 8;
}

template <int M, int KM, int KC, int NB>
__global__ void __launch_bounds__(kThreads, 2) argmax_mma_kernel(const ArgmaxArgs a)
{
    static_assert(M >= 1 && M <= kMaxRows, "one to sixteen hidden rows");
    constexpr bool kHi = M > 8;  // hidden rows 8.. fill the A operand's rows 8..15
    static_assert(KC % kChunk == 0, "the width must be a multiple of the chunk");
    constexpr int CC = KC / kChunk;
    static_assert(CC % NB == 0, "the ring must divide the chunks");
    static_assert(CC > NB, "the second part of h is waited for at chunk NB");
    constexpr int P = pitch<KC>();
    extern __shared__ __align__(16) unsigned char smem[];
    uint16_t *s_h = reinterpret_cast<uint16_t *>(smem);                          // [M][P]
    uint64_t *s_cand = reinterpret_cast<uint64_t *>(smem + (size_t)M * P * 2);   // [M][kLists][KM]

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, q = lane & 3;
    const uint16_t *__restrict__ W = static_cast<const uint16_t *>(a.w);

    // Let the next kernel on the stream start launching its blocks (it waits
    // for this grid before it reads anything this grid writes).
    pdl_launch_dependents();

    // This warp's rows, walked 8 at a time.
    const long long GW = (long long)gridDim.x * kWarps;
    const long long gw = (long long)blockIdx.x * kWarps + warp;
    const int row0 = (int)((long long)a.N * gw / GW);
    const int nrows = (int)((long long)a.N * (gw + 1) / GW) - row0;
    const int ntiles = (nrows + kTile - 1) / kTile;

    // The ring: NB chunks of this lane's two 32-byte pieces of row g, as
    // four 16-byte words (piece w = words 2w, 2w + 1).
    uint4 buf[NB][4];
#pragma unroll
    for (int b = 0; b < NB; ++b)
#pragma unroll
        for (int w = 0; w < 4; ++w)
            buf[b][w] = make_uint4(0u, 0u, 0u, 0u);
    const uint16_t *gp = W + (size_t)(row0 + g) * KC + 16 * q;
    bool vcur = g < nrows;
    auto load_chunk = [&](uint4(&b)[4], const uint16_t *p, int c) {
#pragma unroll
        for (int w = 0; w < 2; ++w)
            ld_stream32(p + kChunk * c + 64 * w, b[2 * w], b[2 * w + 1]);
    };
    auto prologue = [&]() {
        if (vcur) {
#pragma unroll
            for (int c = 0; c < NB; ++c)
                load_chunk(buf[c], gp, c);
        }
    };
    if (a.head_static)
        prologue();
    // From here on: inputs and workspace that earlier work may have written.
    pdl_wait();

    // Copy the hidden rows into shared memory (16-byte asynchronous copies).
    // At width 5,120 in two groups: the k-range of the first NB chunks,
    // which the ring already holds, then the rest, which is waited for only
    // before chunk NB of the first tile, so the MMAs on the buffered chunks
    // overlap the second group's L2 round trip (0.65 us less per call on the
    // 32,768-row trim at 3 and 4 rows; at 2,560 the mid-loop barrier cost
    // more than it saved: +0.9 us at 16 rows on the 52,755-row head).
    constexpr bool kSplit = KC >= 5120;
    {
        constexpr int kA = (kSplit ? NB * kChunk : KC) / 8;  // pieces per row, first group
        for (int i = tid; i < M * kA; i += kThreads) {
            const int m = i / kA, e = 8 * (i - m * kA);
            cp_async16(s_h + m * P + e, a.h + (size_t)m * KC + e);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
        constexpr int kB = KC / 8 - kA;      // the rest of each row
        for (int i = tid; i < M * kB; i += kThreads) {
            const int m = i / kB, e = 8 * (kA + i - m * kB);
            cp_async16(s_h + m * P + e, a.h + (size_t)m * KC + e);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    }
    for (int i = tid; i < M * kLists * KM; i += kThreads)
        s_cand[i] = 0ull;
    if constexpr (kSplit)
        asm volatile("cp.async.wait_group 1;" ::: "memory");
    else
        asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();
    if (!a.head_static)
        prologue();
    // the block-wide wait for the second group: every thread reaches exactly
    // one (here for a warp with no rows, else before chunk NB of tile 0)
    auto rest_of_h = []() {
        asm volatile("cp.async.wait_all;" ::: "memory");
        __syncthreads();
    };
    if (kSplit && ntiles == 0)
        rest_of_h();

    TopList<KM> best;
    best.init();
    // independent accumulators, so consecutive MMAs do not wait on each
    // other; summed at the end of a tile
    float acc[kAcc][4];
#pragma unroll
    for (int i = 0; i < kAcc; ++i)
        acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    const bool hrow = g < M;
    const uint16_t *hp = s_h + (hrow ? g : M - 1) * P + 16 * q;
    const bool hrow2 = kHi && g + 8 < M;  // this lane also ends with hidden row g + 8
    const uint16_t *hp2 = s_h + (hrow2 ? g + 8 : M - 1) * P + 16 * q;
    TopList<KM> best2;
    best2.init();

    for (int t = 0; t < ntiles; ++t) {
        const bool vnext = (t + 1) * kTile + g < nrows;
        // ids of the two rows whose logits this lane ends with
        const int ra = t * kTile + 2 * q;
        int ida = 0, idb = 0;
        if (hrow) {
            if (ra < nrows)
                ida = a.d2t ? __ldg(a.d2t + row0 + ra) : (int)(a.id_base + row0 + ra);
            if (ra + 1 < nrows)
                idb = a.d2t ? __ldg(a.d2t + row0 + ra + 1) : (int)(a.id_base + row0 + ra + 1);
        }
#pragma unroll
        for (int c = 0; c < CC; ++c) {
            const int b = c % NB;
            if (kSplit && c == NB && t == 0)
                rest_of_h();
            // the hidden values of the same k as the lane's words
            uint4 hv[4], hv2[4];
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const int off = kChunk * c + 64 * (w >> 1) + 8 * (w & 1);
                hv[w] = *reinterpret_cast<const uint4 *>(hp + off);
                hv2[w] = kHi ? *reinterpret_cast<const uint4 *>(hp2 + off)
                             : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                mma_bf16(acc[(2 * w) % kAcc], hv[w].x, hv2[w].x, hv[w].y, hv2[w].y, buf[b][w].x,
                         buf[b][w].y);
                mma_bf16(acc[(2 * w + 1) % kAcc], hv[w].z, hv2[w].z, hv[w].w, hv2[w].w,
                         buf[b][w].z, buf[b][w].w);
            }
            const int cn = c + NB;
            if (cn < CC) {
                if (vcur)
                    load_chunk(buf[b], gp, cn);
            } else if (vnext) {
                load_chunk(buf[b], gp + (size_t)kTile * KC, cn - CC);
            }
        }
        float d0 = acc[0][0], d1 = acc[0][1], d2 = acc[0][2], d3 = acc[0][3];
#pragma unroll
        for (int i = 1; i < kAcc; ++i) {
            d0 += acc[i][0];
            d1 += acc[i][1];
            d2 += acc[i][2];
            d3 += acc[i][3];
        }
#pragma unroll
        for (int i = 0; i < kAcc; ++i)
            acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
        if (hrow) {
            if (ra < nrows)
                best.insert(make_key(d0, ida));
            if (ra + 1 < nrows)
                best.insert(make_key(d1, idb));
        }
        if (hrow2) {
            if (ra < nrows)
                best2.insert(make_key(d2, ida));
            if (ra + 1 < nrows)
                best2.insert(make_key(d3, idb));
        }
        gp += (size_t)kTile * KC;
        vcur = vnext;
    }

    if (hrow) {
#pragma unroll
        for (int i = 0; i < KM; ++i)
            s_cand[(g * kLists + warp * 4 + q) * KM + i] = best.v[i];
    }
    if (hrow2) {
#pragma unroll
        for (int i = 0; i < KM; ++i)
            s_cand[((g + 8) * kLists + warp * 4 + q) * KM + i] = best2.v[i];
    }
    __syncthreads();
    block_finish<KM>(s_cand, M, kLists, a);
}

template <int M, int KM, int KC, int NB>
cudaError_t launch(const ArgmaxArgs &a, cudaStream_t s)
{
    const size_t smem = smem_bytes<M, KM, KC>();
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess)
        return e;
    auto kern = argmax_mma_kernel<M, KM, KC, NB>;
    int per_sm = 0;
    e = blocks_per_sm(reinterpret_cast<const void *>(kern), kThreads, smem, &per_sm);
    if (e != cudaSuccess)
        return e;
    if (per_sm < 1)
        return cudaErrorInvalidConfiguration;
    if (per_sm > 2)
        per_sm = 2;
    long long grid = stream_grid(di.sms, per_sm);
    const long long max_by_rows = ((long long)a.N + kWarps - 1) / kWarps;  // >= 1 row per warp
    if (grid > max_by_rows)
        grid = max_by_rows;
    if (grid > kMaxCtas)
        grid = kMaxCtas;
    if (grid < 1)
        grid = 1;
    return launch_pdl(kern, (unsigned)grid, kThreads, smem, s, a);
}

}  // namespace bf16mma
}  // namespace dvl
