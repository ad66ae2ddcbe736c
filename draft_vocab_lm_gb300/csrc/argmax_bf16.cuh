// Fused skinny projection + argmax / top-k over a bf16 draft head, on CUDA
// cores.  One pass streams W once from HBM; the logits live only in
// registers.  ("Shortlist MTP", section "What I was testing": a hidden row of
// width 2,560 against every head row, M = 1 or 3 -- a very wide,
// bandwidth-heavy operation for a couple of rows; sections "What was actually
// happening" / "Re-running the comparison fairly": the skinny low-M kernel and
// the local argmax reduction.)
//
// Work split.  The grid is persistent (two 256-thread blocks per SM).  The N
// rows are cut into one contiguous, balanced range per warp of the whole grid
// (+-1 row).  A warp walks its range RPW rows at a time ("a group"); for each
// group every lane reads 16 bytes (8 weights) of each row per 256-wide k step,
// so one warp load instruction covers 512 contiguous bytes of one row.  Loads
// run NB k steps ahead of the arithmetic through a register ring, across group
// boundaries.  For the hidden widths of the workloads (2,560 and 5,120) K is a
// compile-time constant: the k loop is fully unrolled and every load of a
// group is one base pointer plus an immediate offset, so streaming costs one
// load instruction per 16 bytes and nothing else.  Other widths (multiples
// of 64) take the same kernel with K read at run time.
//
// The hidden rows sit in shared memory as fp32, laid out so that the lane's 8
// values for a k step are two conflict-free 16-byte reads, reused for the RPW
// rows.  At the end of a group the RPW x M partial sums are combined across
// the warp by a reduce-scatter; the lane that ends up owning (row, hidden row)
// forms the packed key (logit, full id) and keeps its best keys.  Each block
// then merges its lanes' lists and the last block to finish merges the
// grid's (block_finish).
#pragma once

#include <cuda_runtime.h>

#include "dvl_device.cuh"

namespace dvl {
namespace bf16 {


constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kKStep = 256;    // weights per row per warp load instruction

// Shared-memory layout of a hidden row (fp32): element e = 256 j + 8 l +
// 4 half + i sits at 256 j + 128 half + 4 l + i, so lane l's 8 values for
// k step j are two conflict-free 16-byte reads.

template <int RPW, int M>
__device__ __forceinline__ void fma_step(float (&acc)[RPW][M], const uint4 (&w)[RPW],
                                         const float *hp, int Kpad)
{
    float wf[RPW][8];
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
        wf[r][0] = bf16_lo(w[r].x); wf[r][1] = bf16_hi(w[r].x);
        wf[r][2] = bf16_lo(w[r].y); wf[r][3] = bf16_hi(w[r].y);
        wf[r][4] = bf16_lo(w[r].z); wf[r][5] = bf16_hi(w[r].z);
        wf[r][6] = bf16_lo(w[r].w); wf[r][7] = bf16_hi(w[r].w);
    }
#pragma unroll
    for (int m = 0; m < M; ++m) {
        const float4 h0 = *reinterpret_cast<const float4 *>(hp + m * Kpad);
        const float4 h1 = *reinterpret_cast<const float4 *>(hp + m * Kpad + 128);
        const float hv[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
#pragma unroll
        for (int r = 0; r < RPW; ++r) {
            float s = acc[r][m];
#pragma unroll
            for (int e = 0; e < 8; ++e)
                s = fmaf(wf[r][e], hv[e], s);
            acc[r][m] = s;
        }
    }
}

// K == KC (a multiple of 256) when KC > 0; K read from the arguments when 0.
template <int M, int KM, int KC, int NB, int RPW>
__global__ void __launch_bounds__(kThreads, 2) argmax_bf16_kernel(const ArgmaxArgs a)
{
    constexpr int kLists = kWarps * RPW;
    extern __shared__ __align__(16) unsigned char smem[];
    const int K = KC > 0 ? KC : a.K;
    const int Kpad = KC > 0 ? KC : a.Kpad;
    const int J = Kpad / kKStep;
    float *s_h = reinterpret_cast<float *>(smem);                       // [M][Kpad]
    uint64_t *s_cand = reinterpret_cast<uint64_t *>(smem + (size_t)M * Kpad * 4);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint16_t *__restrict__ W = static_cast<const uint16_t *>(a.w);

    // Let the next kernel on the stream start launching its blocks as soon as
    // SMs free up (programmatic dependent launch); it waits for this grid's
    // results before it reads anything this grid writes.
    pdl_launch_dependents();

    // This warp's rows.
    const long long GW = (long long)gridDim.x * kWarps;
    const long long gw = (long long)blockIdx.x * kWarps + warp;
    const int row0 = (int)((long long)a.N * gw / GW);
    const int nrows = (int)((long long)a.N * (gw + 1) / GW) - row0;
    const int ngroups = (nrows + RPW - 1) / RPW;

    // The compile-time-K register ring and its first NB k steps.  A head the
    // caller marked static starts streaming before the wait for the
    // preceding kernel on the stream; otherwise after it.
    constexpr int NBc = KC > 0 ? NB : 1;
    uint4 buf[NBc][RPW];
#pragma unroll
    for (int j = 0; j < NBc; ++j)
#pragma unroll
        for (int r = 0; r < RPW; ++r)
            buf[j][r] = make_uint4(0u, 0u, 0u, 0u);
    bool vcur[RPW];
#pragma unroll
    for (int r = 0; r < RPW; ++r)
        vcur[r] = r < nrows;
    const uint16_t *gp = W + (size_t)row0 * (KC > 0 ? KC : 0) + 8 * lane;
    auto prologue = [&]() {
        if constexpr (KC > 0) {
#pragma unroll
            for (int j = 0; j < NB; ++j)
#pragma unroll
                for (int r = 0; r < RPW; ++r)
                    if (vcur[r])
                        buf[j][r] =
                            __ldg(reinterpret_cast<const uint4 *>(gp + r * KC + j * kKStep));
        }
    };
    if (a.head_static)
        prologue();
    // From here on: inputs and workspace that earlier work may have written.
    pdl_wait();

    // Three hidden rows at width 2,560: h is staged in two parts.  The k
    // range of the first NB steps is stored before the main loop; the rest
    // is loaded up front into registers and stored at one block barrier
    // before step NB of the first group, so its stores wait behind the
    // first steps' arithmetic (16,000-row shortlist: 15.7 -> 15.3 us per
    // call; four rows would spill).
    constexpr bool kSplitH = KC == 2560 && M == 3;
    constexpr int kUA = kSplitH ? NB * 32 : 0;  // 16-byte units per row in the first part
    constexpr int kPerB = KC / 8 - kUA;         // and in the rest (used when kSplitH)
    constexpr int kPB = kSplitH ? (M * kPerB + kThreads - 1) / kThreads : 1;
    uint4 vb[kPB];
    auto store_unit = [&](int m, int e, const uint4 &x) {
        float *dst = s_h + m * Kpad + (e & ~255) + ((e & 255) >> 3) * 4;
        *reinterpret_cast<float4 *>(dst) =
            make_float4(bf16_lo(x.x), bf16_hi(x.x), bf16_lo(x.y), bf16_hi(x.y));
        *reinterpret_cast<float4 *>(dst + 128) =
            make_float4(bf16_lo(x.z), bf16_hi(x.z), bf16_lo(x.w), bf16_hi(x.w));
    };
    if constexpr (kSplitH) {
#pragma unroll
        for (int u = 0; u < kPB; ++u) {
            const int i = tid + u * kThreads;
            vb[u] = make_uint4(0u, 0u, 0u, 0u);
            if (i < M * kPerB) {
                const int m = i / kPerB, e = 8 * (kUA + i - m * kPerB);
                vb[u] = __ldg(reinterpret_cast<const uint4 *>(a.h + (size_t)m * K + e));
            }
        }
        for (int i = tid; i < M * kUA; i += kThreads) {
            const int m = i / kUA, e = 8 * (i - m * kUA);
            store_unit(m, e, __ldg(reinterpret_cast<const uint4 *>(a.h + (size_t)m * K + e)));
        }
    }
    // Stage the hidden rows (bf16 -> fp32, zero past K): 16-byte loads, all
    // of a thread's loads issued before its shared-memory stores.
    if constexpr (!kSplitH) {
        constexpr int kMaxPer = 10;  // covers M * Kpad <= 10 * 8 * 256 (four rows of 5,120)
        const int nvec = M * (Kpad / 8);
        uint4 v[kMaxPer];
#pragma unroll
        for (int u = 0; u < kMaxPer; ++u) {
            const int i = tid + u * kThreads;
            v[u] = make_uint4(0u, 0u, 0u, 0u);
            if (i < nvec) {
                const int m = i / (Kpad / 8);
                const int e = 8 * (i - m * (Kpad / 8));
                if (e < K)
                    v[u] = __ldg(reinterpret_cast<const uint4 *>(a.h + (size_t)m * K + e));
            }
        }
#pragma unroll
        for (int u = 0; u < kMaxPer; ++u) {
            const int i = tid + u * kThreads;
            if (i < nvec) {
                const int m = i / (Kpad / 8);
                const int e = 8 * (i - m * (Kpad / 8));
                store_unit(m, e, v[u]);
            }
        }
        for (int i = tid + kMaxPer * kThreads; i < nvec; i += kThreads) {
            const int m = i / (Kpad / 8);
            const int e = 8 * (i - m * (Kpad / 8));
            uint4 x = make_uint4(0u, 0u, 0u, 0u);
            if (e < K)
                x = __ldg(reinterpret_cast<const uint4 *>(a.h + (size_t)m * K + e));
            store_unit(m, e, x);
        }
    }
    for (int i = tid; i < M * kLists * KM; i += kThreads)
        s_cand[i] = 0ull;
    __syncthreads();
    if (!a.head_static)
        prologue();
    // the second part of h; every thread reaches exactly one call (a warp
    // without rows here, the others before step NB of their first group)
    auto rest_of_h = [&]() {
        if constexpr (kSplitH) {
#pragma unroll
            for (int u = 0; u < kPB; ++u) {
                const int i = tid + u * kThreads;
                if (i < M * kPerB) {
                    const int m = i / kPerB, e = 8 * (kUA + i - m * kPerB);
                    store_unit(m, e, vb[u]);
                }
            }
            __syncthreads();
        }
    };
    if (kSplitH && ngroups == 0)
        rest_of_h();

    // Which (row slot, hidden row) this lane owns after the reduce-scatter.
    constexpr int NV = RPW * M;
    constexpr int P = pow2_ceil(NV);
    constexpr int SH = 5 - log2_exact(P);
    const int vi = lane >> SH;
    const bool owner = ((lane & ((1 << SH) - 1)) == 0) && vi < NV;
    const int own_r = vi / M, own_m = vi - (vi / M) * M;

    TopList<KM> best;
    best.init();
    float acc[RPW][M];
#pragma unroll
    for (int r = 0; r < RPW; ++r)
#pragma unroll
        for (int m = 0; m < M; ++m)
            acc[r][m] = 0.f;

    auto finish_group = [&](int g, int pend_id) {
        float v[P];
#pragma unroll
        for (int i = 0; i < P; ++i)
            v[i] = 0.f;
#pragma unroll
        for (int r = 0; r < RPW; ++r)
#pragma unroll
            for (int m = 0; m < M; ++m) {
                v[r * M + m] = acc[r][m];
                acc[r][m] = 0.f;
            }
        warp_reduce_scatter<P>(v);
        if (owner && g * RPW + own_r < nrows)
            best.insert(make_key(v[0], pend_id));
    };
    auto owner_id = [&](int g) {
        int id = 0;
        const int rr = g * RPW + own_r;
        if (owner && rr < nrows) {
            const int row = row0 + rr;
            id = a.d2t ? __ldg(a.d2t + row) : (int)(a.id_base + row);
        }
        return id;
    };

    if constexpr (KC > 0) {
        // ---- compile-time K: unrolled k loop, immediate-offset loads ----
        constexpr int JC = KC / kKStep;
        static_assert(JC % NB == 0, "the ring must divide the k steps");
        for (int g = 0; g < ngroups; ++g) {
            bool vnext[RPW];
#pragma unroll
            for (int r = 0; r < RPW; ++r)
                vnext[r] = (g + 1) * RPW + r < nrows;
            const int pend_id = owner_id(g);
            const float *hp = s_h + lane * 4;
#pragma unroll
            for (int j = 0; j < JC; ++j) {
                const int b = j % NB;
                if (kSplitH && j == NB && g == 0)
                    rest_of_h();
                fma_step<RPW, M>(acc, buf[b], hp + j * kKStep, KC);
                const int jj = j + NB;
#pragma unroll
                for (int r = 0; r < RPW; ++r) {
                    if (jj < JC) {
                        if (vcur[r])
                            buf[b][r] = __ldg(
                                reinterpret_cast<const uint4 *>(gp + r * KC + jj * kKStep));
                    } else if (vnext[r]) {
                        buf[b][r] = __ldg(reinterpret_cast<const uint4 *>(
                            gp + (RPW + r) * KC + (jj - JC) * kKStep));
                    }
                }
            }
            finish_group(g, pend_id);
            gp += RPW * KC;
#pragma unroll
            for (int r = 0; r < RPW; ++r)
                vcur[r] = vnext[r];
        }
    } else {
        // ---- run-time K: one flat (group, k step) stream, predicated ----
        constexpr int NBG = 2;
        const int total = ngroups * J;
        const uint16_t *wlane = W + 8 * lane;
        const bool ktail = (K % kKStep) != 0;
        int ls = 0, lj = 0, cs = 0, cj = 0, pend_id = 0;
        uint4 buf[NBG][RPW];
        auto issue = [&](uint4(&b)[RPW]) {
            const bool kin = !ktail || (lj * kKStep + 8 * lane) < K;
            const uint16_t *p = wlane + (size_t)(row0 + ls * RPW) * K + lj * kKStep;
#pragma unroll
            for (int r = 0; r < RPW; ++r)
                b[r] = (kin && ls * RPW + r < nrows) ? ld_stream16(p + (size_t)r * K)
                                                     : make_uint4(0u, 0u, 0u, 0u);
            if (++lj == J) {
                lj = 0;
                ++ls;
            }
        };
#pragma unroll
        for (int b = 0; b < NBG; ++b)
            issue(buf[b]);
        for (int t0 = 0; t0 < total; t0 += NBG) {
#pragma unroll
            for (int b = 0; b < NBG; ++b) {
                if (t0 + b < total) {
                    if (cj == 0)
                        pend_id = owner_id(cs);
                    fma_step<RPW, M>(acc, buf[b], s_h + cj * kKStep + lane * 4, Kpad);
                    if (++cj == J) {
                        finish_group(cs, pend_id);
                        cj = 0;
                        ++cs;
                    }
                }
                issue(buf[b]);
            }
        }
    }

    if (owner) {
#pragma unroll
        for (int i = 0; i < KM; ++i)
            s_cand[(own_m * kLists + warp * RPW + own_r) * KM + i] = best.v[i];
    }
    __syncthreads();
    block_finish<KM>(s_cand, M, kLists, a);
}

template <int M, int KM, int KC, int NB, int RPW>
cudaError_t launch_cfg(const ArgmaxArgs &a, cudaStream_t s)
{
    const size_t smem = (size_t)M * a.Kpad * 4 + (size_t)M * kWarps * RPW * KM * 8;
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess)
        return e;
    auto kern = argmax_bf16_kernel<M, KM, KC, NB, RPW>;
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
    // A head too short for two full row groups per warp on the full grid:
    // one or two hidden rows at a compile-time width take the smallest grid
    // that gives every warp two full groups, if that keeps at least three
    // quarters of the blocks (measured: the 16,000-row shortlist at one
    // hidden row takes 13.5 instead of 14.0 us on 250 blocks instead of
    // 304; fewer blocks on longer heads were slower).
    if constexpr (KC > 0 && M <= 2) {
        const long long two_groups = (long long)kWarps * 2 * RPW;
        const long long want = ((long long)a.N + two_groups - 1) / two_groups;
        if (want < grid && 4 * want >= 3 * grid)
            grid = want;
    }
    if (grid > kMaxCtas)
        grid = kMaxCtas;
    if (grid < 1)
        grid = 1;
    return launch_pdl(kern, (unsigned)grid, kThreads, smem, s, a);
}

// Per hidden-row count: ring depth and rows per group for each width.
template <int M, int KM>
cudaError_t launch_m(const ArgmaxArgs &a, cudaStream_t s)
{
    static_assert(M <= 4, "5 or more hidden rows run on the tensor cores or in chunks");
    // (Three to eight rows on a long head of width 2,560 or 5,120 never get
    // here: the dispatch sends them to the register-path tensor cores.)
    // Ring depth NB (k steps in flight) and rows per group RPW, chosen by
    // measurement on GB300 among the variants that do not spill at 128
    // registers: a deep ring for M <= 2; for K = 5,120 and M = 3, 4 two rows
    // per group with a 5-deep ring beat four rows with a 2-deep one.
    if (a.K == 2560)
        return launch_cfg<M, KM, 2560, (M <= 2 ? 5 : 2), 4>(a, s);
    if (a.K == 5120) {
        if constexpr (M <= 2)
            return launch_cfg<M, KM, 5120, 5, 4>(a, s);
        else if constexpr (M <= 4)
            return launch_cfg<M, KM, 5120, 5, 2>(a, s);
        else
            return launch_cfg<M, KM, 5120, 2, 4>(a, s);
    }
    // (run-time K, four hidden rows, top-k: two rows per group; four spill)
    if constexpr (M == 4 && KM > 1)
        return launch_cfg<M, KM, 0, 2, 2>(a, s);
    else
        return launch_cfg<M, KM, 0, 2, 4>(a, s);
}

inline int kpad_of(int K) { return (K + kKStep - 1) / kKStep * kKStep; }

}  // namespace bf16
}  // namespace dvl
