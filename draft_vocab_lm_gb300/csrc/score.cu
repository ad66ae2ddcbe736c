// Candidate scoring through a head: for every hidden row m and candidate j,
// the logit of the head row the candidate id names.  ("Masked MTP drafts",
// section "Update (November 2026)": a drafter that carries no head of its
// own scores its candidates through the target's LM head, bf16 or NVFP4,
// and the trim stacks on top; FP8 heads are read the same way.)
//
// A gather-GEMV: the rows are scattered, few (M x c dots) and each is read
// once, so the kernel is bound by memory latency, not bandwidth.  One warp
// computes one dot at a time, taking (m, j) pairs grid-stride:
//   - bf16: lane l covers weights 8 l .. 8 l + 7 of every 256-wide k step;
//     at the unrolled widths (2,560 and 5,120) every 16-byte load of the
//     row is issued before the first multiply, so a dot costs one memory
//     latency; h is read through L1 (every warp of a block reads the same
//     rows);
//   - NVFP4: lane l covers one 16-weight scale block (8 bytes of codes and
//     its E4M3 scale) of every 512-wide k step; codes and scale are decoded
//     exactly (E2M1x2 -> f16x2 -> fp32, E4M3 -> fp32), the block's products
//     (exact in fp32) are summed and multiplied by the block scale, and the
//     tensor scale is applied to the finished dot;
//   - FP8: lane l covers 16 weights (one 16-byte load) of every 512-wide k
//     step, decoded exactly (E4M3x2 -> f16x2 -> fp32), the tensor scale on
//     the finished dot;
//   - the lanes' partial sums meet in a butterfly; lane 0 writes the logit,
//     or NaN when the id is outside the head's rows.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "dvl_device.cuh"

namespace dvl {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ float warp_sum(float x)
{
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1)
        x += __shfl_xor_sync(kFull, x, off);
    return x;
}

__device__ __forceinline__ float dot8_bf16(const uint4 &w, const uint4 &h, float acc)
{
    acc = fmaf(bf16_lo(w.x), bf16_lo(h.x), acc);
    acc = fmaf(bf16_hi(w.x), bf16_hi(h.x), acc);
    acc = fmaf(bf16_lo(w.y), bf16_lo(h.y), acc);
    acc = fmaf(bf16_hi(w.y), bf16_hi(h.y), acc);
    acc = fmaf(bf16_lo(w.z), bf16_lo(h.z), acc);
    acc = fmaf(bf16_hi(w.z), bf16_hi(h.z), acc);
    acc = fmaf(bf16_lo(w.w), bf16_lo(h.w), acc);
    acc = fmaf(bf16_hi(w.w), bf16_hi(h.w), acc);
    return acc;
}

// The head row a pair's id names, or -1 when it is outside the head.
__device__ __forceinline__ long long pair_row(const ScoreArgs &a, long long p)
{
    const long long row = (long long)__ldg(a.ids + p) - a.id_base;
    return (row >= 0 && row < a.N) ? row : -1;
}

// K == KC when KC > 0 (a multiple of 256); K read from the arguments when 0.
template <int KC>
__global__ void __launch_bounds__(kThreads) score_bf16_kernel(const ScoreArgs a)
{
    pdl_launch_dependents();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const long long total = (long long)a.M * a.c;
    const long long GW = (long long)gridDim.x * kWarps;
    const uint16_t *__restrict__ W = static_cast<const uint16_t *>(a.w);
    for (long long p = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5); p < total; p += GW) {
        const int m = (int)(p / a.c);
        const long long row = pair_row(a, p);
        float acc = 0.f;
        if (row >= 0) {
            if constexpr (KC > 0) {
                constexpr int J = KC / 256;
                const uint16_t *wr = W + row * KC + 8 * lane;
                const uint16_t *hr = a.h + (size_t)m * KC + 8 * lane;
                uint4 wv[J];
#pragma unroll
                for (int j = 0; j < J; ++j)
                    wv[j] = ld_stream16(wr + 256 * j);
#pragma unroll
                for (int j = 0; j < J; ++j)
                    acc = dot8_bf16(wv[j], __ldg(reinterpret_cast<const uint4 *>(hr + 256 * j)),
                                    acc);
            } else {
                const int K = a.K;
                const uint16_t *wr = W + row * K;
                const uint16_t *hr = a.h + (size_t)m * K;
#pragma unroll 4
                for (int k0 = 8 * lane; k0 < K; k0 += 256)
                    acc = dot8_bf16(ld_stream16(wr + k0),
                                    __ldg(reinterpret_cast<const uint4 *>(hr + k0)), acc);
            }
        }
        acc = warp_sum(acc);
        if (lane == 0)
            a.out[p] = row >= 0 ? acc : __int_as_float(0x7fc00000);
    }
}

// E4M3 byte -> fp32 (exact) through the hardware f16x2 conversion.
__device__ __forceinline__ float e4m3_to_f32(uint32_t byte)
{
    uint32_t p;
    const uint16_t s = (uint16_t)byte;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(p) : "h"(s));
    return __half2float(__ushort_as_half((unsigned short)(p & 0xffffu)));
}

// 16 codes (8 bytes, low nibble = even k) against 16 hidden values.
__device__ __forceinline__ float dot16_e2m1(uint2 codes, const uint4 &h0, const uint4 &h1)
{
    const uint32_t cw[2] = {codes.x, codes.y};
    const uint32_t hw[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        uint32_t f[4];
        asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
            "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
            "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
            "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
            "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
            "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
            : "=r"(f[0]), "=r"(f[1]), "=r"(f[2]), "=r"(f[3])
            : "r"(cw[i]));
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const float2 w2 = __half22float2(*reinterpret_cast<const __half2 *>(&f[t]));
            const uint32_t hx = hw[4 * i + t];
            acc = fmaf(w2.x, bf16_lo(hx), acc);
            acc = fmaf(w2.y, bf16_hi(hx), acc);
        }
    }
    return acc;
}

__global__ void __launch_bounds__(kThreads) score_nvfp4_kernel(const ScoreArgs a)
{
    pdl_launch_dependents();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const long long total = (long long)a.M * a.c;
    const long long GW = (long long)gridDim.x * kWarps;
    const uint8_t *__restrict__ Q = static_cast<const uint8_t *>(a.w);
    const int K = a.K;
    for (long long p = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5); p < total; p += GW) {
        const int m = (int)(p / a.c);
        const long long row = pair_row(a, p);
        float acc = 0.f;
        if (row >= 0) {
            const uint8_t *qr = Q + row * (K / 2);
            const uint8_t *sr = a.scales + row * (K / 16);
            const uint16_t *hr = a.h + (size_t)m * K;
#pragma unroll 2
            for (int k0 = 16 * lane; k0 < K; k0 += 512) {
                const uint2 codes = __ldg(reinterpret_cast<const uint2 *>(qr + k0 / 2));
                const float s = e4m3_to_f32(__ldg(sr + k0 / 16));
                const uint4 h0 = __ldg(reinterpret_cast<const uint4 *>(hr + k0));
                const uint4 h1 = __ldg(reinterpret_cast<const uint4 *>(hr + k0 + 8));
                acc = fmaf(s, dot16_e2m1(codes, h0, h1), acc);
            }
        }
        acc = warp_sum(acc) * a.gscale;
        if (lane == 0)
            a.out[p] = row >= 0 ? acc : __int_as_float(0x7fc00000);
    }
}

// FP8: lane l covers 16 weights (16 code bytes, one load) of every 512-wide
// k step; E4M3x2 -> f16x2 -> fp32 is exact and so is each product with h.
__global__ void __launch_bounds__(kThreads) score_fp8_kernel(const ScoreArgs a)
{
    pdl_launch_dependents();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const long long total = (long long)a.M * a.c;
    const long long GW = (long long)gridDim.x * kWarps;
    const uint8_t *__restrict__ Q = static_cast<const uint8_t *>(a.w);
    const int K = a.K;
    for (long long p = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5); p < total; p += GW) {
        const int m = (int)(p / a.c);
        const long long row = pair_row(a, p);
        float acc = 0.f;
        if (row >= 0) {
            const uint8_t *qr = Q + row * K;
            const uint16_t *hr = a.h + (size_t)m * K;
#pragma unroll 2
            for (int k0 = 16 * lane; k0 < K; k0 += 512) {
                const uint4 codes = ld_stream16(qr + k0);
                const uint4 h0 = __ldg(reinterpret_cast<const uint4 *>(hr + k0));
                const uint4 h1 = __ldg(reinterpret_cast<const uint4 *>(hr + k0 + 8));
                const uint32_t cw[4] = {codes.x, codes.y, codes.z, codes.w};
                const uint32_t hw[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    uint32_t f0, f1;
                    asm("{\n\t.reg .b16 lo, hi;\n\t"
                        "mov.b32 {lo, hi}, %2;\n\t"
                        "cvt.rn.f16x2.e4m3x2 %0, lo;\n\t"
                        "cvt.rn.f16x2.e4m3x2 %1, hi;\n\t}"
                        : "=r"(f0), "=r"(f1)
                        : "r"(cw[i]));
                    const float2 w0 = __half22float2(*reinterpret_cast<const __half2 *>(&f0));
                    const float2 w1 = __half22float2(*reinterpret_cast<const __half2 *>(&f1));
                    acc = fmaf(w0.x, bf16_lo(hw[2 * i]), acc);
                    acc = fmaf(w0.y, bf16_hi(hw[2 * i]), acc);
                    acc = fmaf(w1.x, bf16_lo(hw[2 * i + 1]), acc);
                    acc = fmaf(w1.y, bf16_hi(hw[2 * i + 1]), acc);
                }
            }
        }
        acc = warp_sum(acc) * a.gscale;
        if (lane == 0)
            a.out[p] = row >= 0 ? acc : __int_as_float(0x7fc00000);
    }
}

}  // namespace

cudaError_t launch_score(const ScoreArgs &a, cudaStream_t s)
{
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess)
        return e;
    const long long pairs = (long long)a.M * a.c;
    long long grid = (pairs + kWarps - 1) / kWarps;
    const long long cap = (long long)di.sms * 8;  // eight blocks per SM at most
    if (grid > cap)
        grid = cap;
    if (grid < 1)
        grid = 1;
    if (a.dtype == DVL_NVFP4)
        return launch_pdl(score_nvfp4_kernel, (unsigned)grid, kThreads, 0, s, a);
    if (a.dtype == DVL_FP8)
        return launch_pdl(score_fp8_kernel, (unsigned)grid, kThreads, 0, s, a);
    if (a.K == 2560)
        return launch_pdl(score_bf16_kernel<2560>, (unsigned)grid, kThreads, 0, s, a);
    if (a.K == 5120)
        return launch_pdl(score_bf16_kernel<5120>, (unsigned)grid, kThreads, 0, s, a);
    return launch_pdl(score_bf16_kernel<0>, (unsigned)grid, kThreads, 0, s, a);
}

}  // namespace dvl
