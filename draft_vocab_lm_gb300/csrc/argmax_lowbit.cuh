// Fused projection + argmax / top-k over a low-bit draft head: NVFP4 or FP8.
// ("Masked MTP drafts": requantizing the trimmed head to NVFP4 costs no
// measured acceptance, and the head read shrinks a further 3.6x against
// bf16; a drafter ships its own FP8 head.  "[DGX Spark] Qwen3.8-Flash-Next
// on two DGX Sparks", section "The costs: a 69% smaller KV pool and FP8 GDN
// weights": weights read as FP8 E4M3 halve the bytes.)
//
// Formats read here (FMT):
//   NVFP4: codes [N][K/2], two E2M1 values per byte with the even k in the
//          low nibble; scales [N][K/16], one E4M3 per 16 consecutive k of a
//          row; one fp32 tensor scale g.  weight = e2m1 * e4m3 * g.
//   FP8:   codes [N][K], one E4M3 per byte; one fp32 tensor scale g.
//          weight = e4m3 * g.
//
// Decoding on CUDA cores costs more instructions per weight than HBM leaves
// time for, so the products run on the tensor cores through the register
// path (mma.sync m16n8k16, f16 inputs, fp32 accumulation), which takes its
// A operand straight from the registers the codes were decoded into:
//   - the grid is persistent (two blocks per SM) and every warp owns one
//     balanced contiguous range of head rows, walked as 16-row MMA tiles
//     (the last one partial); lane (g, q) covers weights 32 q .. 32 q + 31
//     of rows g and g + 8 in every 128-wide k chunk: 16 bytes of NVFP4 codes
//     (two scale blocks) or 32 bytes of FP8 codes per row, so a quad reads
//     one contiguous piece of each row;
//   - a head the caller marked static starts filling the load ring before
//     the wait for the preceding kernel; for the unrolled widths h is read
//     from L2 once (its maximum and its staging from the same registers);
//   - NVFP4: each code byte becomes an f16 pair with the exact E2M1x2 ->
//     f16x2 conversion and is multiplied by its block's E4M3 scale (E4M3x2 ->
//     f16x2); the product has at most 6 significant bits and lies in
//     [2^-10, 2688], so it is exact in f16.  FP8: each pair of code bytes
//     becomes an f16 pair with the exact E4M3x2 -> f16x2 conversion;
//   - the hidden rows are staged once per block as f16 after an exact
//     power-of-two rescale that puts their largest magnitude in [2^14, 2^15)
//     (bf16 values within 2^31 of that maximum convert exactly; smaller ones
//     round at 2^-24 of the rescaled range); the rescale and g are applied to
//     the finished fp32 dot;
//   - the k order inside an MMA is a permutation of the weights' k, the same
//     for A and B, so every product pairs the right weight and hidden value.
// Results go through the same per-lane lists, block merge and cross-block
// finish as the bf16 kernels.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "dvl_device.cuh"

namespace dvl {
namespace lowbit {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRows = 16;      // head rows per warp group (MMA M)
constexpr int kChunk = 128;    // weights per row per k chunk
constexpr int kFmtNvfp4 = 0, kFmtFp8 = 1;
// 16-byte code loads per row per chunk per lane, code bytes per row per
// k chunk, and k chunks of loads in flight per lane: 4 (measured against 2
// and 5; ~4.5 KB per warp for NVFP4, ~8 KB for FP8).  Top-k keeps its
// lists in shared memory, so it affords the same ring as argmax.
template <int FMT> __host__ __device__ constexpr int q_words() { return FMT == kFmtFp8 ? 2 : 1; }
template <int FMT> __host__ __device__ constexpr int chunk_bytes() { return FMT == kFmtFp8 ? 128 : 64; }
template <int FMT, int M, int KC, int KM>
__host__ __device__ constexpr int ring_depth()
{
    // FP8 argmax with four hidden rows at 5,120 spills registers with a
    // 4-deep ring (ptxas); a 2-deep one keeps it within 128
    return (FMT == kFmtFp8 && M >= 4 && KC == 5120 && KM == 1) ? 2 : 4;
}
constexpr int kLists = kWarps * 8;  // candidate lists per hidden row (8 row pairs per warp)

// Four bytes of codes -> four f16x2 (byte t: low nibble in the low half).
__device__ __forceinline__ void e2m1_word(uint32_t w, uint32_t (&f)[4])
{
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(f[0]), "=r"(f[1]), "=r"(f[2]), "=r"(f[3])
        : "r"(w));
}

// Two E4M3 scales (low byte first) -> f16x2, and each broadcast to a pair.
__device__ __forceinline__ void e4m3_pair(uint32_t s16, uint32_t &lo2, uint32_t &hi2)
{
    uint32_t p;
    const uint16_t s = (uint16_t)s16;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(p) : "h"(s));
    lo2 = __byte_perm(p, p, 0x1010);
    hi2 = __byte_perm(p, p, 0x3232);
}

// Four bytes of E4M3 codes -> two f16x2 (bytes 0, 1 and 2, 3; the lower
// byte in the low half).
__device__ __forceinline__ void e4m3_word(uint32_t w, uint32_t &f0, uint32_t &f1)
{
    asm("{\n\t.reg .b16 lo, hi;\n\t"
        "mov.b32 {lo, hi}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, lo;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, hi;\n\t}"
        : "=r"(f0), "=r"(f1)
        : "r"(w));
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ void mma_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float pow2f(int e)  // 2^e for e in [-126, 127], exact
{
    return __int_as_float((127 + e) << 23);
}

// Shared memory: the rescaled hidden rows as f16, in 16-byte units ordered
// [chunk][u][g][q] with g < M (unit = h[g][128 chunk + 32 q + 8 u .. +8]), so
// that the reading lanes' units for one u are contiguous.  Lanes whose MMA
// column g is M or more feed zeros and read nothing.
__host__ __device__ inline size_t lowbit_h_bytes(int Kpad, int M) { return (size_t)Kpad * 2 * M; }

// K == KC (a multiple of 128) when KC > 0; K read from the arguments when 0.
template <int FMT, int M, int KM, int KC>
__global__ void __launch_bounds__(kThreads, 2) argmax_lowbit_kernel(const ArgmaxArgs a)
{
    constexpr int kNB = ring_depth<FMT, M, KC, KM>(), kQW = q_words<FMT>();
    constexpr bool kNv = FMT == kFmtNvfp4;
    extern __shared__ __align__(16) unsigned char smem[];
    const int K = KC > 0 ? KC : a.K;
    const int Kpad = KC > 0 ? KC : a.Kpad, C = Kpad / kChunk;
    uint4 *s_h = reinterpret_cast<uint4 *>(smem);
    uint64_t *s_cand = reinterpret_cast<uint64_t *>(smem + lowbit_h_bytes(Kpad, M));
    __shared__ unsigned int s_wmax[kWarps];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, q = lane & 3;
    const uint8_t *__restrict__ Q = static_cast<const uint8_t *>(a.w);
    const uint8_t *__restrict__ S = a.scales;
    const size_t qrow = kNv ? (size_t)K / 2 : (size_t)K, srow = (size_t)K / 16;

    pdl_launch_dependents();

    // This warp's rows: one balanced contiguous range per warp of the grid,
    // walked 16 rows (one MMA tile) at a time; the last group may be partial.
    const long long GW = (long long)gridDim.x * kWarps;
    const long long gw = (long long)blockIdx.x * kWarps + warp;
    const int row0 = (int)((long long)a.N * gw / GW);
    const int rend = (int)((long long)a.N * (gw + 1) / GW);
    const int my_groups = (rend - row0 + kRows - 1) / kRows;

    // The load ring: codes (16 or 32 bytes) and, for NVFP4, scales (two
    // E4M3) of rows ra / rb.
    uint4 bqa[kNB][kQW], bqb[kNB][kQW];
    uint32_t bsa[kNB], bsb[kNB];
#pragma unroll
    for (int b2 = 0; b2 < kNB; ++b2) {
#pragma unroll
        for (int w = 0; w < kQW; ++w)
            bqa[b2][w] = bqb[b2][w] = make_uint4(0u, 0u, 0u, 0u);
        bsa[b2] = bsb[b2] = 0u;
    }
    // compile-time K: a group's lane bases, codes of rows ra / rb at byte
    // 16 q (NVFP4) or 32 q (FP8), scales at 2 q; loads are immediate offsets
    constexpr int QR = kNv ? KC / 2 : KC, SR = KC / 16;  // bytes per row: codes, scales
    constexpr int CB = chunk_bytes<FMT>();
    auto bases = [&](int li, const uint8_t *&pqa, const uint8_t *&psa, bool &va, bool &vb) {
        const int ra = row0 + li * kRows + g;
        va = li < my_groups && ra < rend;
        vb = li < my_groups && ra + 8 < rend;
        pqa = Q + (size_t)ra * QR + 16 * kQW * q;
        psa = S + (size_t)ra * SR + 2 * q;
    };
    auto load = [&](int b2, const uint8_t *pqa, const uint8_t *psa, bool va, bool vb, int c) {
        if (va) {
#pragma unroll
            for (int w = 0; w < kQW; ++w)
                bqa[b2][w] = ld_stream16(pqa + CB * c + 16 * w);
            if constexpr (kNv)
                bsa[b2] = __ldg(reinterpret_cast<const unsigned short *>(psa + 8 * c));
        }
        if (vb) {
#pragma unroll
            for (int w = 0; w < kQW; ++w)
                bqb[b2][w] = ld_stream16(pqa + 8 * QR + CB * c + 16 * w);
            if constexpr (kNv)
                bsb[b2] = __ldg(reinterpret_cast<const unsigned short *>(psa + 8 * SR + 8 * c));
        }
    };
    const uint8_t *pqa = Q, *psa = S;
    bool va = false, vb = false;
    auto prologue = [&]() {
        if constexpr (KC > 0) {
            bases(0, pqa, psa, va, vb);
#pragma unroll
            for (int c = 0; c < kNB; ++c)
                load(c, pqa, psa, va, vb, c);
        }
    };
    // A head the caller marked static starts streaming before the wait for
    // the preceding kernel on the stream; otherwise after it.
    if (a.head_static)
        prologue();
    pdl_wait();

    // Stage h as f16, scaled by 2^shift so that max|h| * 2^shift lies in
    // [2^14, 2^15): hmax = f * 2^e with f in [0.5, 1), e = bf16 exponent
    // field - 126 (bf16 magnitudes order like their bit patterns).
    auto shift_of = [](unsigned int hmax) {
        const int ef = (int)(hmax >> 7);
        const int sh = hmax == 0u ? 0 : (ef == 0 ? 100 : 15 - (ef - 126));
        return min(max(sh, -100), 100);
    };
    auto to_f16 = [](const uint4 &x, float up) {
        const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
        uint32_t hv[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const __half2 hh = __floats2half2_rn(bf16_lo(xs[j]) * up, bf16_hi(xs[j]) * up);
            hv[j] = *reinterpret_cast<const uint32_t *>(&hh);
        }
        return make_uint4(hv[0], hv[1], hv[2], hv[3]);
    };
    auto block_max = [&](unsigned int mx) {
        for (int off = 16; off >= 1; off >>= 1)
            mx = max(mx, __shfl_xor_sync(kFull, mx, off));
        if (lane == 0)
            s_wmax[warp] = mx;
    };
    auto read_max = [&]() {
        unsigned int mx = 0u;
#pragma unroll
        for (int w = 0; w < kWarps; ++w)
            mx = max(mx, s_wmax[w]);
        return mx;
    };
    // unit i = h[gg][k0 .. k0 + 8], ordered [chunk][u][g][q] (see above)
    auto unit_k0 = [](int i, int &gg) {
        const int qq = i & 3, r = i >> 2;
        gg = r % M;
        const int u = (r / M) & 3, c = r / (M * 4);
        return kChunk * c + 32 * qq + 8 * u;
    };
    int shift;
    for (int i = tid; i < M * kLists * KM; i += kThreads)
        s_cand[i] = 0ull;
    if constexpr (KC > 0) {
        // one pass: every unit loaded once, its maximum taken, then stored
        constexpr int kUnits = (KC / kChunk) * 16 * M;
        constexpr int kPer = (kUnits + kThreads - 1) / kThreads;
        uint4 hx[kPer];
        unsigned int mx = 0u;
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            const int i = tid + j * kThreads;
            hx[j] = make_uint4(0u, 0u, 0u, 0u);
            if (i < kUnits) {
                int gg;
                const int k0 = unit_k0(i, gg);
                hx[j] = __ldg(reinterpret_cast<const uint4 *>(a.h + (size_t)gg * KC + k0));
            }
        }
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            const uint32_t xs[4] = {hx[j].x, hx[j].y, hx[j].z, hx[j].w};
#pragma unroll
            for (int t = 0; t < 4; ++t)
                mx = max(mx, max(xs[t] & 0x7fffu, (xs[t] >> 16) & 0x7fffu));
        }
        block_max(mx);
        __syncthreads();
        shift = shift_of(read_max());
        const float up = shift >= 0 ? pow2f(min(shift, 127)) : pow2f(max(shift, -126));
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            const int i = tid + j * kThreads;
            if (i < kUnits)
                s_h[i] = to_f16(hx[j], up);
        }
    } else {
        // two passes over h from L2: the maximum, then the staging
        unsigned int mx = 0u;
        for (int i = tid; i < M * K / 2; i += kThreads) {
            const uint32_t x = __ldg(reinterpret_cast<const uint32_t *>(a.h) + i);
            mx = max(mx, max(x & 0x7fffu, (x >> 16) & 0x7fffu));
        }
        block_max(mx);
        __syncthreads();
        shift = shift_of(read_max());
        const float up = shift >= 0 ? pow2f(min(shift, 127)) : pow2f(max(shift, -126));
        const int nunits = C * 4 * M * 4;
        for (int i = tid; i < nunits; i += kThreads) {
            int gg;
            const int k0 = unit_k0(i, gg);
            uint4 x = make_uint4(0u, 0u, 0u, 0u);
            if (k0 < K)
                x = __ldg(reinterpret_cast<const uint4 *>(a.h + (size_t)gg * K + k0));
            s_h[i] = to_f16(x, up);
        }
    }
    __syncthreads();
    if (!a.head_static)
        prologue();
    const float down = (shift >= 0 ? pow2f(max(-shift, -126)) : pow2f(min(-shift, 127))) * a.gscale;

    // argmax: the best key of hidden rows 2q and 2q + 1 in registers; top-k:
    // the lists in this lane's own candidate slots in shared memory (zeroed
    // above), which the block merge reads at the end
    TopList<1> best0, best1;
    best0.init();
    best1.init();
    const int slot = warp * 8 + g;
    uint64_t *list0 = s_cand + ((size_t)(2 * q) * kLists + slot) * KM;
    uint64_t *list1 = s_cand + ((size_t)(2 * q + 1) * kLists + slot) * KM;
    auto keep0 = [&](uint64_t key) {
        if constexpr (KM == 1)
            best0.insert(key);
        else
            list_insert_smem<KM>(list0, key);
    };
    auto keep1 = [&](uint64_t key) {
        if constexpr (KM == 1)
            best1.insert(key);
        else
            list_insert_smem<KM>(list1, key);
    };
    // four independent accumulators, so consecutive MMAs do not wait on
    // each other; summed at the end of a group
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    // B fragments: lanes whose MMA column g >= M keep zeros throughout
    uint32_t hw[16];
#pragma unroll
    for (int j = 0; j < 16; ++j)
        hw[j] = 0u;

    // One 128-wide k chunk of rows ra (codes qa, scales sa) and rb.
    auto chunk = [&](const uint4 (&qa)[kQW], const uint4 (&qb)[kQW], uint32_t sa, uint32_t sb,
                     int cidx) {
        if (g < M) {
            const uint4 *hp = s_h + (size_t)cidx * (16 * M) + (g * 4 + q);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const uint4 v = hp[u * 4 * M];
                hw[4 * u] = v.x; hw[4 * u + 1] = v.y; hw[4 * u + 2] = v.z; hw[4 * u + 3] = v.w;
            }
        }
        if constexpr (!kNv) {
            // FP8: code word t (k = 32 q + 4 t .. + 3) of each row is exactly
            // the A operand of MMA t: decode it as it is used
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                const uint4 &xa = qa[t >> 2], &xb = qb[t >> 2];
                const uint32_t wa = (t & 3) == 0 ? xa.x : (t & 3) == 1 ? xa.y : (t & 3) == 2 ? xa.z : xa.w;
                const uint32_t wb = (t & 3) == 0 ? xb.x : (t & 3) == 1 ? xb.y : (t & 3) == 2 ? xb.z : xb.w;
                uint32_t a0, a2, a1, a3;
                e4m3_word(wa, a0, a2);
                e4m3_word(wb, a1, a3);
                mma_f16(acc[t & 3], a0, a1, a2, a3, hw[2 * t], hw[2 * t + 1]);
            }
            return;
        }
        // fa[i], fb[i]: the f16 pair of k = 32 q + 2 i, + 1 of rows ra, rb
        uint32_t fa[16], fb[16];
        if constexpr (kNv) {
            uint32_t sa_lo, sa_hi, sb_lo, sb_hi;
            e4m3_pair(sa, sa_lo, sa_hi);
            e4m3_pair(sb, sb_lo, sb_hi);
            const uint32_t wa[4] = {qa[0].x, qa[0].y, qa[0].z, qa[0].w};
            const uint32_t wb[4] = {qb[0].x, qb[0].y, qb[0].z, qb[0].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t t4[4];
                e2m1_word(wa[j], t4);
                fa[4 * j] = t4[0]; fa[4 * j + 1] = t4[1]; fa[4 * j + 2] = t4[2]; fa[4 * j + 3] = t4[3];
                e2m1_word(wb[j], t4);
                fb[4 * j] = t4[0]; fb[4 * j + 1] = t4[1]; fb[4 * j + 2] = t4[2]; fb[4 * j + 3] = t4[3];
            }
            // the block scale: k < 32 q + 16 uses the lower scale byte
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                fa[i] = hmul2(fa[i], i < 8 ? sa_lo : sa_hi);
                fb[i] = hmul2(fb[i], i < 8 ? sb_lo : sb_hi);
            }
        }
#pragma unroll
        for (int t = 0; t < 8; ++t)
            mma_f16(acc[t & 3], fa[2 * t], fb[2 * t], fa[2 * t + 1], fb[2 * t + 1], hw[2 * t],
                    hw[2 * t + 1]);
    };
    // Rows ra (c0, c1) and rb (c2, c3) of a finished group; hidden rows 2q, 2q + 1.
    auto finish_group = [&](int ra, int ida, int idb) {
        const int rb = ra + 8;
        float d[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            d[j] = (acc[0][j] + acc[1][j]) + (acc[2][j] + acc[3][j]);
            acc[0][j] = acc[1][j] = acc[2][j] = acc[3][j] = 0.f;
        }
        if (ra < rend) {
            if (2 * q < M)
                keep0(make_key(d[0] * down, ida));
            if (2 * q + 1 < M)
                keep1(make_key(d[1] * down, ida));
        }
        if (rb < rend) {
            if (2 * q < M)
                keep0(make_key(d[2] * down, idb));
            if (2 * q + 1 < M)
                keep1(make_key(d[3] * down, idb));
        }
    };
    auto row_id = [&](int r) {
        return r < rend ? (a.d2t ? __ldg(a.d2t + r) : (int)(a.id_base + r)) : 0;
    };

    if constexpr (KC > 0) {
        // ---- compile-time K: one base pointer per group, immediate offsets ----
        constexpr int CC = KC / kChunk;
        static_assert(CC % kNB == 0, "the ring must divide the chunks");
        // NVFP4 unrolls the whole group; FP8 (twice the code bytes per
        // chunk) a multiple of the ring, which keeps it within the registers
        constexpr int kCU = kNv ? CC : 2 * kNB;
        for (int li = 0; li < my_groups; ++li) {
            const uint8_t *nqa, *nsa;
            bool nva, nvb;
            bases(li + 1, nqa, nsa, nva, nvb);
            const int ra = row0 + li * kRows + g;
            const int ida = row_id(ra), idb = row_id(ra + 8);
#pragma unroll(kCU)
            for (int c = 0; c < CC; ++c) {
                const int b2 = c % kNB;
                chunk(bqa[b2], bqb[b2], bsa[b2], bsb[b2], c);
                if (c + kNB < CC)
                    load(b2, pqa, psa, va, vb, c + kNB);
                else
                    load(b2, nqa, nsa, nva, nvb, c + kNB - CC);
            }
            finish_group(ra, ida, idb);
            pqa = nqa;
            psa = nsa;
            va = nva;
            vb = nvb;
        }
    } else {
        // ---- run-time K: one flat (group, chunk) stream, predicated ----
        const int total = my_groups * C;
        int li = 0, lc = 0;  // load cursor (my group index, chunk)
        auto issue = [&](int b2) {
            const int ra = row0 + li * kRows + g, rb = ra + 8;
            const int kc = kChunk * lc + 32 * q;
            const bool kin = li < my_groups && kc < K;  // K % 64 == 0: all 32 k in range
            const size_t cb = kNv ? (size_t)kc / 2 : (size_t)kc;  // code byte of k = kc
#pragma unroll
            for (int w = 0; w < kQW; ++w)
                bqa[b2][w] = bqb[b2][w] = make_uint4(0u, 0u, 0u, 0u);
            bsa[b2] = 0u;
            bsb[b2] = 0u;
            if (kin && ra < rend) {
#pragma unroll
                for (int w = 0; w < kQW; ++w)
                    bqa[b2][w] = ld_stream16(Q + (size_t)ra * qrow + cb + 16 * w);
                if constexpr (kNv)
                    bsa[b2] = __ldg(reinterpret_cast<const unsigned short *>(
                        S + (size_t)ra * srow + kc / 16));
            }
            if (kin && rb < rend) {
#pragma unroll
                for (int w = 0; w < kQW; ++w)
                    bqb[b2][w] = ld_stream16(Q + (size_t)rb * qrow + cb + 16 * w);
                if constexpr (kNv)
                    bsb[b2] = __ldg(reinterpret_cast<const unsigned short *>(
                        S + (size_t)rb * srow + kc / 16));
            }
            if (++lc == C) {
                lc = 0;
                ++li;
            }
        };
        int ci = 0, cc = 0, ida = 0, idb = 0;
#pragma unroll
        for (int b2 = 0; b2 < kNB; ++b2)
            issue(b2);
        for (int t0 = 0; t0 < total; t0 += kNB) {
#pragma unroll
            for (int b2 = 0; b2 < kNB; ++b2) {
                if (t0 + b2 < total) {
                    const int ra = row0 + ci * kRows + g;
                    if (cc == 0) {
                        ida = row_id(ra);
                        idb = row_id(ra + 8);
                    }
                    chunk(bqa[b2], bqb[b2], bsa[b2], bsb[b2], cc);
                    if (++cc == C) {
                        finish_group(ra, ida, idb);
                        cc = 0;
                        ++ci;
                    }
                }
                issue(b2);
            }
        }
    }

    if constexpr (KM == 1) {
        if (2 * q < M)
            list0[0] = best0.v[0];
        if (2 * q + 1 < M)
            list1[0] = best1.v[0];
    }
    __syncthreads();
    block_finish<KM>(s_cand, M, kLists, a);
}

template <int FMT, int M, int KM, int KC>
cudaError_t launch_one(const ArgmaxArgs &a, cudaStream_t s)
{
    const size_t smem = lowbit_h_bytes(a.Kpad, M) + (size_t)M * kLists * KM * 8;
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess)
        return e;
    auto kern = argmax_lowbit_kernel<FMT, M, KM, KC>;
    int per_sm = 0;
    e = blocks_per_sm(reinterpret_cast<const void *>(kern), kThreads, smem, &per_sm);
    if (e != cudaSuccess)
        return e;
    if (per_sm < 1)
        return cudaErrorInvalidConfiguration;
    if (per_sm > 2)
        per_sm = 2;
    long long grid = (long long)di.sms * per_sm;
    // at least half an MMA tile of rows per warp on average
    const long long max_by_rows = ((long long)a.N + kWarps * 8 - 1) / (kWarps * 8);
    if (grid > max_by_rows)
        grid = max_by_rows;
    if (grid > kMaxCtas)
        grid = kMaxCtas;
    if (grid < 1)
        grid = 1;
    return launch_pdl(kern, (unsigned)grid, kThreads, smem, s, a);
}

inline int kpad_of(int K) { return (K + kChunk - 1) / kChunk * kChunk; }

template <int FMT, int KM, int KC>
cudaError_t dispatch_m(const ArgmaxArgs &a, int M, cudaStream_t s)
{
    switch (M) {
    case 1: return launch_one<FMT, 1, KM, KC>(a, s);
    case 2: return launch_one<FMT, 2, KM, KC>(a, s);
    case 3: return launch_one<FMT, 3, KM, KC>(a, s);
    case 4: return launch_one<FMT, 4, KM, KC>(a, s);
    case 5: return launch_one<FMT, 5, KM, KC>(a, s);
    case 6: return launch_one<FMT, 6, KM, KC>(a, s);
    case 7: return launch_one<FMT, 7, KM, KC>(a, s);
    case 8: return launch_one<FMT, 8, KM, KC>(a, s);
    default: return cudaErrorInvalidValue;
    }
}

// argmax (KM = 1) or top-k (KM = 4) at the unrolled widths (K = 2,560 or
// 5,120, M <= 4): one base pointer per group with immediate offsets.
template <int FMT, int KM>
cudaError_t launch_kc(const ArgmaxArgs &a, int M, cudaStream_t s)
{
    if (a.K == 5120) {
        switch (M) {
        case 1: return launch_one<FMT, 1, KM, 5120>(a, s);
        case 2: return launch_one<FMT, 2, KM, 5120>(a, s);
        case 3: return launch_one<FMT, 3, KM, 5120>(a, s);
        case 4: return launch_one<FMT, 4, KM, 5120>(a, s);
        }
    } else if (a.K == 2560) {
        switch (M) {
        case 1: return launch_one<FMT, 1, KM, 2560>(a, s);
        case 2: return launch_one<FMT, 2, KM, 2560>(a, s);
        case 3: return launch_one<FMT, 3, KM, 2560>(a, s);
        case 4: return launch_one<FMT, 4, KM, 2560>(a, s);
        }
    }
    return cudaErrorInvalidValue;
}

// argmax / top-k with K read at run time, M <= 8.
template <int FMT>
cudaError_t launch_rt(const ArgmaxArgs &a, int M, int kmax, cudaStream_t s)
{
    return kmax == 1 ? dispatch_m<FMT, 1, 0>(a, M, s) : dispatch_m<FMT, 4, 0>(a, M, s);
}

// Each format's instantiations live in a translation unit of their own
// (compiled in parallel).
extern template cudaError_t launch_kc<kFmtNvfp4, 1>(const ArgmaxArgs &, int, cudaStream_t);
extern template cudaError_t launch_kc<kFmtFp8, 1>(const ArgmaxArgs &, int, cudaStream_t);
extern template cudaError_t launch_kc<kFmtNvfp4, 4>(const ArgmaxArgs &, int, cudaStream_t);
extern template cudaError_t launch_kc<kFmtFp8, 4>(const ArgmaxArgs &, int, cudaStream_t);
extern template cudaError_t launch_rt<kFmtNvfp4>(const ArgmaxArgs &, int, int, cudaStream_t);
extern template cudaError_t launch_rt<kFmtFp8>(const ArgmaxArgs &, int, int, cudaStream_t);

}  // namespace lowbit
}  // namespace dvl
