// Fused projection + argmax / top-k over an NVFP4 draft head, on CUDA cores.
// ("Masked MTP drafts": requantizing the trimmed head to NVFP4 costs no
// measured acceptance; the head read shrinks a further 3.6x against bf16.)
//
// Format read here: codes [N][K/2], two E2M1 values per byte with the even k
// in the low nibble; scales [N][K/16], one E4M3 per 16 consecutive k of a
// row; one fp32 tensor scale g.  weight = e2m1 * e4m3 * g.
//
// The structure follows the bf16 kernel (per-warp balanced row ranges, RPW
// rows per group, loads NBUF k-steps ahead, reduce-scatter, packed keys,
// block and grid merges).  A lane reads 16 bytes of codes (32 weights, two
// scale blocks) and the 2 scale bytes of those blocks per row per k step; a
// warp load instruction covers 512 contiguous bytes of codes.  The codes are
// widened with the hardware E2M1x2 -> f16x2 conversion (exact), each 16-wide
// block is summed in fp32 against the fp32 hidden values, then scaled by its
// E4M3 block scale (E4M3x2 -> f16x2, exact); g multiplies the finished dot.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "dvl_device.cuh"

namespace dvl {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRPW = 4;
constexpr int kNBuf = 2;
constexpr int kKStep = 1024;   // weights per row per warp load instruction
static_assert(kWarps * kRPW == 32, "block_finish expects 32 lists per hidden row");

// Shared-memory offset of hidden element e = 1024 j + 32 l + 8 w + 4 half + i
// (word w of lane l's 32 weights): 1024 j + 256 w + 128 half + 4 l + i.
__device__ __forceinline__ int h_slot(int e)
{
    return (e & ~1023) + ((e >> 3) & 3) * 256 + ((e >> 2) & 1) * 128 + ((e >> 5) & 31) * 4 +
           (e & 3);
}

// Eight E2M1 codes (one 32-bit word, element 2t in the low nibble of byte t)
// to fp32, exactly.
__device__ __forceinline__ void e2m1x8(uint32_t w, float (&f)[8])
{
    uint32_t p0, p1, p2, p3;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(p0), "=r"(p1), "=r"(p2), "=r"(p3)
        : "r"(w));
    const uint32_t p[4] = {p0, p1, p2, p3};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        __half2 hh = *reinterpret_cast<const __half2 *>(&p[t]);
        float2 ff = __half22float2(hh);
        f[2 * t] = ff.x;
        f[2 * t + 1] = ff.y;
    }
}

// Two E4M3 scales (low byte first) to fp32, exactly.
__device__ __forceinline__ float2 e4m3x2(uint32_t s16)
{
    uint32_t p;
    uint16_t s = (uint16_t)s16;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(p) : "h"(s));
    __half2 hh = *reinterpret_cast<const __half2 *>(&p);
    return __half22float2(hh);
}

template <int M, int KM>
__global__ void __launch_bounds__(kThreads, 2) argmax_nvfp4_kernel(const ArgmaxArgs a)
{
    extern __shared__ __align__(16) unsigned char smem[];
    float *s_h = reinterpret_cast<float *>(smem);
    uint64_t *s_cand = reinterpret_cast<uint64_t *>(smem + (size_t)M * a.Kpad * 4);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int K = a.K, Kpad = a.Kpad, J = Kpad / kKStep;
    const uint8_t *__restrict__ Q = static_cast<const uint8_t *>(a.w);
    const uint8_t *__restrict__ S = a.scales;
    const int qrow = K / 2, srow = K / 16;

    for (int i = tid; i < M * (Kpad / 2); i += kThreads) {
        const int m = i / (Kpad / 2);
        const int e = 2 * (i - m * (Kpad / 2));
        uint32_t x = 0u;
        if (e < K)
            x = __ldg(reinterpret_cast<const uint32_t *>(a.h + (size_t)m * K + e));
        float *dst = s_h + m * Kpad + h_slot(e);
        dst[0] = bf16_lo(x);
        dst[1] = bf16_hi(x);
    }
    __syncthreads();

    const long long GW = (long long)gridDim.x * kWarps;
    const long long gw = (long long)blockIdx.x * kWarps + warp;
    const int row0 = (int)((long long)a.N * gw / GW);
    const int nrows = (int)((long long)a.N * (gw + 1) / GW) - row0;
    const int nsteps = (nrows + kRPW - 1) / kRPW;
    const int total = nsteps * J;

    constexpr int NV = kRPW * M;
    constexpr int P = pow2_ceil(NV);
    constexpr int SH = 5 - log2_exact(P);
    const int vi = lane >> SH;
    const bool owner = ((lane & ((1 << SH) - 1)) == 0) && vi < NV;
    const int own_r = vi / M, own_m = vi - (vi / M) * M;

    TopList<KM> best;
    best.init();
    float acc[kRPW][M];
#pragma unroll
    for (int r = 0; r < kRPW; ++r)
#pragma unroll
        for (int m = 0; m < M; ++m)
            acc[r][m] = 0.f;

    const bool ktail = (K % kKStep) != 0;
    int ls = 0, lj = 0, cs = 0, cj = 0;
    int pend_id = 0;

    uint4 qb[kNBuf][kRPW];
    uint32_t sb[kNBuf][kRPW];

    auto issue = [&](uint4(&q)[kRPW], uint32_t(&sc)[kRPW]) {
        const int e0 = lj * kKStep + 32 * lane;
        const bool kin = !ktail || e0 < K;
        const size_t r0 = (size_t)(row0 + ls * kRPW);
#pragma unroll
        for (int r = 0; r < kRPW; ++r) {
            if (kin && ls * kRPW + r < nrows) {
                q[r] = ld_stream16(Q + (r0 + r) * qrow + e0 / 2);
                sc[r] = __ldg(reinterpret_cast<const unsigned short *>(S + (r0 + r) * srow +
                                                                       e0 / 16));
            } else {
                q[r] = make_uint4(0u, 0u, 0u, 0u);
                sc[r] = 0u;
            }
        }
        if (++lj == J) {
            lj = 0;
            ++ls;
        }
    };

    auto consume = [&](const uint4(&q)[kRPW], const uint32_t(&sc)[kRPW]) {
        if (cj == 0 && owner) {
            const int rr = cs * kRPW + own_r;
            if (rr < nrows) {
                const int row = row0 + rr;
                pend_id = a.d2t ? __ldg(a.d2t + row) : (int)(a.id_base + row);
            }
        }
        float2 scale[kRPW];
#pragma unroll
        for (int r = 0; r < kRPW; ++r)
            scale[r] = e4m3x2(sc[r]);
        const float *hp = s_h + cj * kKStep + lane * 4;
        float blk[kRPW][M];
#pragma unroll
        for (int wd = 0; wd < 4; ++wd) {
            float hv[M][8];
#pragma unroll
            for (int m = 0; m < M; ++m) {
                const float4 h0 = *reinterpret_cast<const float4 *>(hp + m * Kpad + 256 * wd);
                const float4 h1 =
                    *reinterpret_cast<const float4 *>(hp + m * Kpad + 256 * wd + 128);
                hv[m][0] = h0.x; hv[m][1] = h0.y; hv[m][2] = h0.z; hv[m][3] = h0.w;
                hv[m][4] = h1.x; hv[m][5] = h1.y; hv[m][6] = h1.z; hv[m][7] = h1.w;
            }
#pragma unroll
            for (int r = 0; r < kRPW; ++r) {
                const uint32_t word = wd == 0 ? q[r].x : wd == 1 ? q[r].y : wd == 2 ? q[r].z : q[r].w;
                float f[8];
                e2m1x8(word, f);
#pragma unroll
                for (int m = 0; m < M; ++m) {
                    float s = (wd & 1) ? blk[r][m] : 0.f;
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        s = fmaf(f[i], hv[m][i], s);
                    blk[r][m] = s;
                }
            }
            if (wd & 1) {
#pragma unroll
                for (int r = 0; r < kRPW; ++r) {
                    const float s = (wd == 1) ? scale[r].x : scale[r].y;
#pragma unroll
                    for (int m = 0; m < M; ++m)
                        acc[r][m] = fmaf(blk[r][m], s, acc[r][m]);
                }
            }
        }
        if (++cj == J) {
            float v[P];
#pragma unroll
            for (int i = 0; i < P; ++i)
                v[i] = 0.f;
#pragma unroll
            for (int r = 0; r < kRPW; ++r)
#pragma unroll
                for (int m = 0; m < M; ++m) {
                    v[r * M + m] = acc[r][m];
                    acc[r][m] = 0.f;
                }
            warp_reduce_scatter<P>(v);
            if (owner && cs * kRPW + own_r < nrows)
                best.insert(make_key(v[0] * a.gscale, pend_id));
            cj = 0;
            ++cs;
        }
    };

#pragma unroll
    for (int b = 0; b < kNBuf; ++b)
        issue(qb[b], sb[b]);
    for (int t0 = 0; t0 < total; t0 += kNBuf) {
#pragma unroll
        for (int b = 0; b < kNBuf; ++b) {
            if (t0 + b < total)
                consume(qb[b], sb[b]);
            issue(qb[b], sb[b]);
        }
    }

    for (int i = tid; i < M * 32 * KM; i += kThreads)
        s_cand[i] = 0ull;
    __syncthreads();
    if (owner) {
#pragma unroll
        for (int i = 0; i < KM; ++i)
            s_cand[(own_m * 32 + warp * kRPW + own_r) * KM + i] = best.v[i];
    }
    __syncthreads();
    block_finish<KM>(s_cand, M, 32, a);
}

template <int M, int KM>
cudaError_t launch_one(const ArgmaxArgs &a, cudaStream_t s)
{
    const size_t smem = (size_t)M * a.Kpad * 4 + (size_t)M * 32 * KM * 8;
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess)
        return e;
    int per_sm = 0;
    e = blocks_per_sm(reinterpret_cast<const void *>(argmax_nvfp4_kernel<M, KM>), kThreads, smem, &per_sm);
    if (e != cudaSuccess)
        return e;
    if (per_sm < 1)
        return cudaErrorInvalidConfiguration;
    if (per_sm > 2)
        per_sm = 2;
    long long grid = (long long)di.sms * per_sm;
    // at least one row per warp
    const long long max_by_rows = ((long long)a.N + kWarps - 1) / kWarps;
    if (grid > max_by_rows)
        grid = max_by_rows;
    if (grid > kMaxCtas)
        grid = kMaxCtas;
    if (grid < 1)
        grid = 1;
    argmax_nvfp4_kernel<M, KM><<<(unsigned)grid, kThreads, smem, s>>>(a);
    return cudaGetLastError();
}

template <int KM>
cudaError_t dispatch_m(const ArgmaxArgs &a, int M, cudaStream_t s)
{
    switch (M) {
    case 1: return launch_one<1, KM>(a, s);
    case 2: return launch_one<2, KM>(a, s);
    case 3: return launch_one<3, KM>(a, s);
    case 4: return launch_one<4, KM>(a, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

int max_chunk_rows_nvfp4(int K)
{
    const int Kpad = (K + kKStep - 1) / kKStep * kKStep;
    int r = (96 * 1024) / (Kpad * 4);
    return r > 4 ? 4 : r;
}

cudaError_t launch_argmax_nvfp4(const ArgmaxArgs &a_in, int M, int kmax, cudaStream_t s)
{
    ArgmaxArgs a = a_in;
    a.Kpad = (a.K + kKStep - 1) / kKStep * kKStep;
    return kmax == 1 ? dispatch_m<1>(a, M, s) : dispatch_m<4>(a, M, s);
}

}  // namespace dvl
