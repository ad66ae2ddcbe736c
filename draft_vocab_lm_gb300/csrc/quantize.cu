// Load-time requantization of a bf16 head to NVFP4 or FP8.  ("Masked MTP
// drafts": the trimmed head requantized to NVFP4 at load costs no measured
// acceptance and shrinks the head read a further 3.6x.)
//
// The recipe (the pages give none; this is the plainest reading), in fp32
// with each operation rounded once, in this order:
//   NVFP4: g = amax / (6 * 448); per 16-weight block s = RNE_e4m3(amax_b /
//          (6 g)); code = RNE_e2m1(w / (s g)); all codes 0 when s is 0.
//   FP8:   g = amax / 448; code = RNE_e4m3(w / g).
// RNE is the hardware round-to-nearest-even conversion with saturation to
// the format's largest finite value (cvt.rn.satfinite); the sign of a code
// is the sign of its quotient.
//
// Two kernels: the head's largest magnitude (16-byte loads grid-stride, a
// warp maximum, one atomicMax per warp on the order-preserving bit pattern)
// into a spare word of the caller's workspace, then - once the host has read
// it and formed g - one thread per 16 consecutive weights: 32 bytes of bf16
// in, 8 bytes of NVFP4 codes plus one scale byte, or 16 bytes of FP8 codes,
// out.  The second kernel clears the workspace word again.
#include <cstring>

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "dvl_device.cuh"

namespace dvl {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) amax_kernel(const uint4 *__restrict__ w, long long n16,
                                                        unsigned int *amax_bits)
{
    unsigned int m = 0u;
    const long long stride = (long long)gridDim.x * kThreads;
    for (long long i = (long long)blockIdx.x * kThreads + threadIdx.x; i < n16; i += stride) {
        const uint4 v = ld_stream16(w + i);
        const uint32_t x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
            m = max(m, max(x[j] & 0x7fffu, (x[j] >> 16) & 0x7fffu));  // bf16 magnitudes
    }
    m = (unsigned int)warp_max_u64(m);
    if ((threadIdx.x & 31) == 0 && m != 0u)
        atomicMax(amax_bits, m << 16);  // the fp32 bit pattern of the bf16 magnitude
}

__device__ __forceinline__ void load16(const uint16_t *src, float (&x)[16])
{
    const uint4 v0 = ld_stream16(src), v1 = ld_stream16(src + 8);
    const uint32_t u[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        x[2 * j] = bf16_lo(u[j]);
        x[2 * j + 1] = bf16_hi(u[j]);
    }
}

// Two fp32 values -> two E4M3 bytes, lo in the low byte (RNE, saturating).
__device__ __forceinline__ uint32_t e4m3x2_rn(float lo, float hi)
{
    uint16_t p;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(p) : "f"(hi), "f"(lo));
    return p;
}

__device__ __forceinline__ float e4m3_value(uint32_t byte)
{
    uint32_t p;
    const uint16_t s = (uint16_t)byte;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(p) : "h"(s));
    return __half2float(__ushort_as_half((unsigned short)(p & 0xffffu)));
}

// Eight fp32 values -> four bytes of E2M1 codes, value 2i in the low nibble
// of byte i (RNE, saturating).
__device__ __forceinline__ uint32_t e2m1x8_rn(const float *x)
{
    uint32_t r;
    asm("{\n\t.reg .b8 t0, t1, t2, t3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t3, %8, %7;\n\t"
        "mov.b32 %0, {t0, t1, t2, t3};\n\t}"
        : "=r"(r)
        : "f"(x[0]), "f"(x[1]), "f"(x[2]), "f"(x[3]), "f"(x[4]), "f"(x[5]), "f"(x[6]),
          "f"(x[7]));
    return r;
}

__global__ void __launch_bounds__(kThreads)
    quantize_nvfp4_kernel(const uint16_t *__restrict__ w, long long nblocks, float g,
                          uint8_t *__restrict__ codes, uint8_t *__restrict__ scales,
                          unsigned int *amax_bits)
{
    if (blockIdx.x == 0 && threadIdx.x == 0)
        *amax_bits = 0u;  // read by the host before this launch: leave the workspace clean
    const float six_g = __fmul_rn(6.0f, g);
    const long long stride = (long long)gridDim.x * kThreads;
    for (long long b = (long long)blockIdx.x * kThreads + threadIdx.x; b < nblocks; b += stride) {
        float x[16];
        load16(w + b * 16, x);
        float amax_b = 0.f;
#pragma unroll
        for (int j = 0; j < 16; ++j)
            amax_b = fmaxf(amax_b, fabsf(x[j]));
        const uint32_t sb = e4m3x2_rn(__fdiv_rn(amax_b, six_g), 0.f) & 0xffu;
        const float s_val = e4m3_value(sb);
        const float sg = __fmul_rn(s_val, g);
        uint2 out = make_uint2(0u, 0u);
        if (s_val != 0.f) {
            float y[16];
#pragma unroll
            for (int j = 0; j < 16; ++j)
                y[j] = __fdiv_rn(x[j], sg);
            out.x = e2m1x8_rn(y);
            out.y = e2m1x8_rn(y + 8);
        }
        *reinterpret_cast<uint2 *>(codes + b * 8) = out;
        scales[b] = (uint8_t)sb;
    }
}

__global__ void __launch_bounds__(kThreads)
    quantize_fp8_kernel(const uint16_t *__restrict__ w, long long nblocks, float g,
                        uint8_t *__restrict__ codes, unsigned int *amax_bits)
{
    if (blockIdx.x == 0 && threadIdx.x == 0)
        *amax_bits = 0u;
    const long long stride = (long long)gridDim.x * kThreads;
    for (long long b = (long long)blockIdx.x * kThreads + threadIdx.x; b < nblocks; b += stride) {
        float x[16];
        load16(w + b * 16, x);
        uint32_t h[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            h[j] = e4m3x2_rn(__fdiv_rn(x[2 * j], g), __fdiv_rn(x[2 * j + 1], g));
        *reinterpret_cast<uint4 *>(codes + b * 16) =
            make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16),
                       h[6] | (h[7] << 16));
    }
}

}  // namespace

cudaError_t launch_quantize(const uint16_t *w, long long n, int dtype, uint8_t *codes,
                            uint8_t *scales, unsigned char *ws, cudaStream_t s, float *g_out)
{
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess)
        return e;
    unsigned int *amax_bits = reinterpret_cast<unsigned int *>(ws + kWsAmax);
    const long long n16 = n / 8;  // 16-byte vectors of bf16
    long long grid = (n16 + kThreads - 1) / kThreads;
    if (grid > (long long)di.sms * 8)
        grid = (long long)di.sms * 8;
    amax_kernel<<<(unsigned)(grid < 1 ? 1 : grid), kThreads, 0, s>>>(
        reinterpret_cast<const uint4 *>(w), n16, amax_bits);
    if ((e = cudaGetLastError()) != cudaSuccess)
        return e;
    unsigned int bits = 0u;
    if ((e = cudaMemcpyAsync(&bits, amax_bits, sizeof bits, cudaMemcpyDeviceToHost, s)) !=
        cudaSuccess)
        return e;
    if ((e = cudaStreamSynchronize(s)) != cudaSuccess)
        return e;
    float amax;
    std::memcpy(&amax, &bits, sizeof amax);
    const float g = amax > 0.f ? amax / (dtype == DVL_NVFP4 ? 2688.0f : 448.0f) : 1.0f;
    const long long nblocks = n / 16;
    grid = (nblocks + kThreads - 1) / kThreads;
    if (grid > (long long)di.sms * 8)
        grid = (long long)di.sms * 8;
    if (grid < 1)
        grid = 1;
    if (dtype == DVL_NVFP4)
        quantize_nvfp4_kernel<<<(unsigned)grid, kThreads, 0, s>>>(w, nblocks, g, codes, scales,
                                                                  amax_bits);
    else
        quantize_fp8_kernel<<<(unsigned)grid, kThreads, 0, s>>>(w, nblocks, g, codes, amax_bits);
    if ((e = cudaGetLastError()) != cudaSuccess)
        return e;
    *g_out = g;
    return cudaSuccess;
}

}  // namespace dvl
