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
//     [2^-10, 2688], so it is exact in f16.  With one hidden row the MMA's
//     eight columns carry the chunk's eight scale blocks instead, and the
//     scales multiply the fp32 block dots (see chunk()).  FP8: each pair
//     of code bytes becomes an f16 pair with the exact E4M3x2 -> f16x2
//     conversion;
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

constexpr int kThreads = 256;  // threads per block when two blocks fit per SM
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
    // FP8 argmax from four hidden rows on spills registers with a 4-deep
    // ring (ptxas), a 2-deep one keeps it within 128; FP8 top-k above 8 rows
    // (lists in shared memory) affords 5, measured 27% faster than 2
    if (M > 8)
        return FMT == kFmtFp8 ? (KM == 1 ? 2 : 5) : 4;
    return (FMT == kFmtFp8 && M >= 4 && KM == 1) ? 2 : 4;
}
constexpr int kLists = kWarps * 8;  // candidate lists per hidden row (8 row pairs per warp)

// Hidden rows are the MMA's n8 columns: ceil(M / 8) groups of 8, each an
// MMA of its own against the same decoded head fragment.
template <int M> __host__ __device__ constexpr int n_groups() { return (M + 7) / 8; }
// Threads per block: 256 (two blocks per SM) unless the staged hidden rows
// (M x K f16) leave room for one block per SM only; then one block of 512.
template <int M, int KC> __host__ __device__ constexpr int block_threads()
{
    return (size_t)M * KC * 2 > 96 * 1024 ? 512 : 256;
}

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

// The same MMA with a zero accumulator in.
__device__ __forceinline__ void mma_f16_zero(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                             uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
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
__global__ void __launch_bounds__(block_threads<M, KC>(), 512 / block_threads<M, KC>())
    argmax_lowbit_kernel(const ArgmaxArgs a)
{
    constexpr int TH = block_threads<M, KC>(), NW = TH / 32, NL = NW * 8;
    constexpr int NG = n_groups<M>();
    // hidden rows of this launch: M itself up to 8; the instantiations for
    // 16 and 32 take any count up to that from a.m_rows
    const int MR = M > 8 ? a.m_rows : M;
    constexpr int kNB = ring_depth<FMT, M, KC, KM>(), kQW = q_words<FMT>();
    constexpr bool kNv = FMT == kFmtNvfp4;
    extern __shared__ __align__(16) unsigned char smem[];
    const int K = KC > 0 ? KC : a.K;
    const int Kpad = KC > 0 ? KC : a.Kpad, C = Kpad / kChunk;
    uint4 *s_h = reinterpret_cast<uint4 *>(smem);
    uint64_t *s_cand = reinterpret_cast<uint64_t *>(smem + lowbit_h_bytes(Kpad, M));
    __shared__ unsigned int s_wmax[NW];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, q = lane & 3;
    const uint8_t *__restrict__ Q = static_cast<const uint8_t *>(a.w);
    const uint8_t *__restrict__ S = a.scales;
    const size_t qrow = kNv ? (size_t)K / 2 : (size_t)K, srow = (size_t)K / 16;

    pdl_launch_dependents();

    // This warp's rows: one balanced contiguous range per warp of the grid,
    // walked 16 rows (one MMA tile) at a time; the last group may be partial.
    const long long GW = (long long)gridDim.x * NW;
    const long long gw = (long long)blockIdx.x * NW + warp;
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
        for (int w = 0; w < NW; ++w)
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
    // unit i of h in h's own order (row gg, elements e .. e + 8) -> its slot
    // in the [chunk][u][g][q] layout (compile-time width)
    auto natural_unit = [](int i, int &gg, int &slot) {
        constexpr int kU = (KC > 0 ? KC : 8) / 8;  // units per row (used with KC > 0)
        gg = i / kU;
        const int e = 8 * (i - gg * kU);
        const int c = e / kChunk, r = e - c * kChunk;
        slot = ((c * 4 + ((r & 31) >> 3)) * M + gg) * 4 + (r >> 5);
        return e;
    };
    int shift;
    for (int i = tid; i < M * NL * KM; i += TH)
        s_cand[i] = 0ull;
    if constexpr (KC > 0 && NG > 1) {
        // many hidden rows: the raw units are copied to shared memory in
        // rounds of four per thread (16-byte loads, then stores; the load
        // ring holds most registers; rows past MR stay zero), read in h's
        // own order so that a warp reads 512 contiguous bytes, each placed
        // at its unit's slot; the maximum is taken from the registers on the
        // way, and each thread then converts its units in place.  (cp.async
        // copies instead: 36.9 against 32.8 us for NVFP4 32,768 x 5,120 at
        // 16 rows, 145.1 against 137.1 for FP8 248,320 x 2,560 at 32.)
        constexpr int kUnits = (KC / kChunk) * 16 * M;
        constexpr int kRound = 4;
        unsigned int mx = 0u;  // the maximum, from the registers as they are stored
        for (int i0 = 0; i0 < kUnits; i0 += kRound * TH) {
            uint4 v[kRound];
            int sl[kRound];
#pragma unroll
            for (int u = 0; u < kRound; ++u) {
                const int i = i0 + u * TH + tid;
                v[u] = make_uint4(0u, 0u, 0u, 0u);
                sl[u] = -1;
                if (i < kUnits) {
                    int gg;
                    const int e = natural_unit(i, gg, sl[u]);
                    if (gg < MR)
                        v[u] = __ldg(reinterpret_cast<const uint4 *>(a.h + (size_t)gg * KC + e));
                }
            }
#pragma unroll
            for (int u = 0; u < kRound; ++u)
                if (sl[u] >= 0) {
                    s_h[sl[u]] = v[u];
                    const uint32_t xs[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
                    for (int t = 0; t < 4; ++t)
                        mx = max(mx, max(xs[t] & 0x7fffu, (xs[t] >> 16) & 0x7fffu));
                }
        }
        block_max(mx);
        __syncthreads();  // units land in other threads' slots; the warp maxima
        shift = shift_of(read_max());
        const float up = shift >= 0 ? pow2f(min(shift, 127)) : pow2f(max(shift, -126));
        for (int i = tid; i < kUnits; i += TH)
            s_h[i] = to_f16(s_h[i], up);  // this thread's own unit
    } else if constexpr (KC > 0) {
        // one pass: every unit loaded once (in h's own order, so a warp reads
        // 512 contiguous bytes), its maximum taken, then stored to its slot
        constexpr int kUnits = (KC / kChunk) * 16 * M;
        constexpr int kPer = (kUnits + TH - 1) / TH;
        uint4 hx[kPer];
        unsigned int mx = 0u;
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            const int i = tid + j * TH;
            hx[j] = make_uint4(0u, 0u, 0u, 0u);
            if (i < kUnits)
                hx[j] = __ldg(reinterpret_cast<const uint4 *>(a.h) + i);  // h is [M][KC]
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
            const int i = tid + j * TH;
            if (i < kUnits) {
                int gg, slot;
                natural_unit(i, gg, slot);
                s_h[slot] = to_f16(hx[j], up);
            }
        }
    } else {
        // two passes over h from L2: the maximum, then the staging
        unsigned int mx = 0u;
        for (int i = tid; i < M * K / 2; i += TH) {
            const uint32_t x = __ldg(reinterpret_cast<const uint32_t *>(a.h) + i);
            mx = max(mx, max(x & 0x7fffu, (x >> 16) & 0x7fffu));
        }
        block_max(mx);
        __syncthreads();
        shift = shift_of(read_max());
        const float up = shift >= 0 ? pow2f(min(shift, 127)) : pow2f(max(shift, -126));
        const int nunits = C * 4 * M * 4;
        for (int i = tid; i < nunits; i += TH) {
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

    // argmax: the best key of hidden rows 8G + 2q and 8G + 2q + 1 (group G)
    // in registers; top-k: the lists in this lane's own candidate slots in
    // shared memory (zeroed above), which the block merge reads at the end
    // (more than one group: the argmax keys live in the shared-memory lists
    // too, which frees the registers)
    constexpr bool kRegBest = KM == 1 && NG == 1;
    TopList<1> best[kRegBest ? 1 : 1][2];
    best[0][0].init();
    best[0][1].init();
    const int slot = warp * 8 + g;
    auto list_of = [&](int m) { return s_cand + ((size_t)m * NL + slot) * KM; };
    auto keep = [&](int G, int s, uint64_t key) {
        if constexpr (kRegBest)
            best[0][s].insert(key);
        else
            list_insert_smem<KM>(list_of(8 * G + 2 * q + s), key);
    };
    // independent accumulator chains (four for one group of hidden rows, two
    // or one per group for more), so consecutive MMAs do not wait on each
    // other; summed at the end of a row group
    constexpr int CH = NG == 1 ? 4 : (NG == 2 ? 2 : 1);
    float acc[NG][CH][4];
#pragma unroll
    for (int G = 0; G < NG; ++G)
#pragma unroll
        for (int i = 0; i < CH; ++i)
            acc[G][i][0] = acc[G][i][1] = acc[G][i][2] = acc[G][i][3] = 0.f;
    // B fragments: lanes whose MMA column g >= M keep zeros throughout
    uint32_t hw[16];
#pragma unroll
    for (int j = 0; j < 16; ++j)
        hw[j] = 0u;

    // One 128-wide k chunk of rows ra (codes qa, scales sa) and rb, against
    // two or more groups of hidden rows: each 16-byte unit of h (pairs 4u ..
    // 4u + 3, i.e. MMAs 2u and 2u + 1) is read per group just before use.
    auto chunk_groups = [&](const uint4 (&qa)[kQW], const uint4 (&qb)[kQW], uint32_t sa,
                            uint32_t sb, int cidx) {
        const uint4 *hp0 = s_h + (size_t)cidx * (16 * M) + q;
        auto hunit = [&](int G, int u) {
            const int gg = 8 * G + g;
            return gg < M ? hp0[u * 4 * M + gg * 4] : make_uint4(0u, 0u, 0u, 0u);
        };
        if constexpr (!kNv) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                uint32_t af[2][4];  // A fragments of MMAs 2u and 2u + 1
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    const int t = 2 * u + h2;
                    const uint4 &xa = qa[t >> 2], &xb = qb[t >> 2];
                    const uint32_t wa = (t & 3) == 0 ? xa.x : (t & 3) == 1 ? xa.y : (t & 3) == 2 ? xa.z : xa.w;
                    const uint32_t wb = (t & 3) == 0 ? xb.x : (t & 3) == 1 ? xb.y : (t & 3) == 2 ? xb.z : xb.w;
                    e4m3_word(wa, af[h2][0], af[h2][2]);
                    e4m3_word(wb, af[h2][1], af[h2][3]);
                }
#pragma unroll
                for (int G = 0; G < NG; ++G) {
                    const uint4 v = hunit(G, u);
                    mma_f16(acc[G][(2 * u) % CH], af[0][0], af[0][1], af[0][2], af[0][3], v.x, v.y);
                    mma_f16(acc[G][(2 * u + 1) % CH], af[1][0], af[1][1], af[1][2], af[1][3], v.z,
                            v.w);
                }
            }
            return;
        }
        // NVFP4: code word u of each row holds pairs 4u .. 4u + 3 (MMAs 2u
        // and 2u + 1); it is decoded and scaled just before its MMAs
        uint32_t sa_lo, sa_hi, sb_lo, sb_hi;
        e4m3_pair(sa, sa_lo, sa_hi);
        e4m3_pair(sb, sb_lo, sb_hi);
        const uint32_t wa[4] = {qa[0].x, qa[0].y, qa[0].z, qa[0].w};
        const uint32_t wb[4] = {qb[0].x, qb[0].y, qb[0].z, qb[0].w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            uint32_t fa[4], fb[4];
            e2m1_word(wa[u], fa);
            e2m1_word(wb[u], fb);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                fa[i] = hmul2(fa[i], u < 2 ? sa_lo : sa_hi);
                fb[i] = hmul2(fb[i], u < 2 ? sb_lo : sb_hi);
            }
#pragma unroll
            for (int G = 0; G < NG; ++G) {
                const uint4 v = hunit(G, u);
                mma_f16(acc[G][(2 * u) % CH], fa[0], fb[0], fa[1], fb[1], v.x, v.y);
                mma_f16(acc[G][(2 * u + 1) % CH], fa[2], fb[2], fa[3], fb[3], v.z, v.w);
            }
        }
    };
    // One 128-wide k chunk of rows ra (codes qa, scales sa) and rb.
    auto chunk = [&](const uint4 (&qa)[kQW], const uint4 (&qb)[kQW], uint32_t sa, uint32_t sb,
                     int cidx) {
        if constexpr (NG > 1) {
            chunk_groups(qa, qb, sa, sb, cidx);
            return;
        }
        if constexpr (kNv && M == 1) {
            // One hidden row: the MMA's eight columns take the chunk's eight
            // scale blocks instead.  MMA t pairs quad position q with k = 32 q
            // + 4 t .. + 3 of both rows, which lie in block 2 q (t < 4) or
            // 2 q + 1 (t >= 4); B puts h there in column 2 q or 2 q + 1 (the
            // lanes g = 2 q, resp. 2 q + 1, hold it; every other B entry
            // stays zero), so result column n is block n's dot of the
            // unscaled codes.  Lane (g, q) holds columns 2 q, 2 q + 1 of rows
            // g and g + 8: exactly the blocks its own two scale bytes per row
            // cover, applied to the fp32 results (4 FMAs per chunk instead of
            // 32 f16x2 multiplies).  The four lanes of a quad hold disjoint
            // blocks of a row: summed at the end of the row group.
            const uint4 *hp = s_h + (size_t)cidx * 16 + q;
            if (g == 2 * q) {
                const uint4 v0 = hp[0], v1 = hp[4];
                hw[0] = v0.x; hw[1] = v0.y; hw[2] = v0.z; hw[3] = v0.w;
                hw[4] = v1.x; hw[5] = v1.y; hw[6] = v1.z; hw[7] = v1.w;
            } else if (g == 2 * q + 1) {
                const uint4 v2 = hp[8], v3 = hp[12];
                hw[8] = v2.x; hw[9] = v2.y; hw[10] = v2.z; hw[11] = v2.w;
                hw[12] = v3.x; hw[13] = v3.y; hw[14] = v3.z; hw[15] = v3.w;
            }
            const uint32_t wa[4] = {qa[0].x, qa[0].y, qa[0].z, qa[0].w};
            const uint32_t wb[4] = {qb[0].x, qb[0].y, qb[0].z, qb[0].w};
            float p[2][4];  // two chains (MMAs t even / odd)
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                uint32_t fa4[4], fb4[4];
                e2m1_word(wa[u], fa4);
                e2m1_word(wb[u], fb4);
                if (u == 0) {
                    mma_f16_zero(p[0], fa4[0], fb4[0], fa4[1], fb4[1], hw[0], hw[1]);
                    mma_f16_zero(p[1], fa4[2], fb4[2], fa4[3], fb4[3], hw[2], hw[3]);
                } else {
                    mma_f16(p[0], fa4[0], fb4[0], fa4[1], fb4[1], hw[4 * u], hw[4 * u + 1]);
                    mma_f16(p[1], fa4[2], fb4[2], fa4[3], fb4[3], hw[4 * u + 2], hw[4 * u + 3]);
                }
            }
            uint32_t s2a, s2b;  // E4M3 pairs -> f16x2 (block 2 q low, 2 q + 1 high)
            asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(s2a) : "h"((uint16_t)sa));
            asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(s2b) : "h"((uint16_t)sb));
            const __half2 ha = *reinterpret_cast<const __half2 *>(&s2a);
            const __half2 hb = *reinterpret_cast<const __half2 *>(&s2b);
            float(&c)[4] = acc[0][cidx & 3];
            c[0] = fmaf(__low2float(ha), p[0][0] + p[1][0], c[0]);
            c[0] = fmaf(__high2float(ha), p[0][1] + p[1][1], c[0]);
            c[2] = fmaf(__low2float(hb), p[0][2] + p[1][2], c[2]);
            c[2] = fmaf(__high2float(hb), p[0][3] + p[1][3], c[2]);
            return;
        }
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
                mma_f16(acc[0][t & 3], a0, a1, a2, a3, hw[2 * t], hw[2 * t + 1]);
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
            mma_f16(acc[0][t & 3], fa[2 * t], fb[2 * t], fa[2 * t + 1], fb[2 * t + 1], hw[2 * t],
                    hw[2 * t + 1]);
    };
    // Rows ra (c0, c1) and rb (c2, c3) of a finished row group; hidden rows
    // 8G + 2q, 8G + 2q + 1 of each group G.
    auto finish_group = [&](int ra, int ida, int idb) {
        const int rb = ra + 8;
#pragma unroll
        for (int G = 0; G < NG; ++G) {
            float d[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if constexpr (CH == 4)
                    d[j] = (acc[G][0][j] + acc[G][1][j]) + (acc[G][2][j] + acc[G][3][j]);
                else if constexpr (CH == 2)
                    d[j] = acc[G][0][j] + acc[G][1][j];
                else
                    d[j] = acc[G][0][j];
#pragma unroll
                for (int c = 0; c < CH; ++c)
                    acc[G][c][j] = 0.f;
            }
            if constexpr (kNv && M == 1 && NG == 1) {
                // one hidden row: the quad's four lanes hold disjoint blocks
#pragma unroll
                for (int j = 0; j < 4; j += 2) {
                    d[j] += __shfl_xor_sync(kFull, d[j], 1);
                    d[j] += __shfl_xor_sync(kFull, d[j], 2);
                }
            }
            const int m0 = 8 * G + 2 * q;
            if (ra < rend) {
                if (m0 < MR)
                    keep(G, 0, make_key(d[0] * down, ida));
                if (m0 + 1 < MR)
                    keep(G, 1, make_key(d[1] * down, ida));
            }
            if (rb < rend) {
                if (m0 < MR)
                    keep(G, 0, make_key(d[2] * down, idb));
                if (m0 + 1 < MR)
                    keep(G, 1, make_key(d[3] * down, idb));
            }
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
        // (more than one group of hidden rows: the same window as FP8)
        constexpr int kCU = kNv && NG == 1 ? CC : 2 * kNB;
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

    if constexpr (kRegBest) {
#pragma unroll
        for (int s2 = 0; s2 < 2; ++s2)
            if (2 * q + s2 < MR)
                list_of(2 * q + s2)[0] = best[0][s2].v[0];
    }
    __syncthreads();
    block_finish<KM>(s_cand, MR, NL, a);
}

template <int FMT, int M, int KM, int KC>
cudaError_t launch_one(const ArgmaxArgs &a, cudaStream_t s)
{
    constexpr int TH = block_threads<M, KC>(), NW = TH / 32;
    const size_t smem = lowbit_h_bytes(a.Kpad, M) + (size_t)M * (NW * 8) * KM * 8;
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess)
        return e;
    auto kern = argmax_lowbit_kernel<FMT, M, KM, KC>;
    int per_sm = 0;
    e = blocks_per_sm(reinterpret_cast<const void *>(kern), TH, smem, &per_sm);
    if (e != cudaSuccess)
        return e;
    if (per_sm < 1)
        return cudaErrorInvalidConfiguration;
    if (per_sm > 512 / TH)
        per_sm = 512 / TH;
    long long grid = stream_grid(di.sms, per_sm);
    // at least half an MMA tile of rows per warp on average
    const long long max_by_rows = ((long long)a.N + NW * 8 - 1) / (NW * 8);
    if (grid > max_by_rows)
        grid = max_by_rows;
    if (grid > kMaxCtas)
        grid = kMaxCtas;
    if (grid < 1)
        grid = 1;
    return launch_pdl(kern, (unsigned)grid, TH, smem, s, a);
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

// argmax / top-k for 9 .. 32 hidden rows in one pass at the unrolled widths:
// instantiated for 16 and 32 rows (two and four groups of 8 MMA columns),
// with the launch's row count in a.m_rows; rows past it stage zeros and are
// not merged.  At 5,120 32 staged rows do not fit, nor do 32 rows of top-k
// lists next to them at 2,560: those calls take 16 rows per launch.
template <int FMT, int KM>
cudaError_t launch_groups(const ArgmaxArgs &a, int M, cudaStream_t s)
{
    ArgmaxArgs b = a;
    b.m_rows = M;
    if (a.K == 2560) {
        if (M <= 16)
            return launch_one<FMT, 16, KM, 2560>(b, s);
        if constexpr (KM == 1)
            return launch_one<FMT, 32, KM, 2560>(b, s);
    }
    if (a.K == 5120 && M <= 16)
        return launch_one<FMT, 16, KM, 5120>(b, s);
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
extern template cudaError_t launch_groups<kFmtNvfp4, 1>(const ArgmaxArgs &, int, cudaStream_t);
extern template cudaError_t launch_groups<kFmtNvfp4, 4>(const ArgmaxArgs &, int, cudaStream_t);
extern template cudaError_t launch_groups<kFmtFp8, 1>(const ArgmaxArgs &, int, cudaStream_t);
extern template cudaError_t launch_groups<kFmtFp8, 4>(const ArgmaxArgs &, int, cudaStream_t);
extern template cudaError_t launch_rt<kFmtFp8>(const ArgmaxArgs &, int, int, cudaStream_t);

}  // namespace lowbit
}  // namespace dvl
