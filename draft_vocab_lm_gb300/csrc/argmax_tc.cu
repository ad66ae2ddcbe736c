// Fused skinny projection + argmax / top-k on the tensor cores (tcgen05, TMEM) for
// batched drafting: 5 to 32 hidden rows at once ("[DGX Spark]
// Qwen3.8-Flash-Next on two DGX Sparks", section "Five changes in 16 days":
// MTP with 4 draft slots, 8 concurrent streams; "Shortlist MTP", section
// "At first, the shortlist looked REALLY good": 8 concurrent requests).  With
// M of 16-32 the projection does 16-32 flops per head byte, more than the
// CUDA cores sustain at HBM rate, so the products go to the tensor cores and
// the kernel stays bound by the one pass over the head.
//
// D[n][m] = sum_k W[n][k] h[m][k] is computed as a 128 x NM tile per 128 head
// rows (A = W tile, K-major; B = h, K-major; NM = 16 or 32 >= M), fp32 in
// tensor memory.  One block of 8 warps per SM, each on a contiguous range of
// rows split into 128-row tiles:
//   warp 0   TMA producer: per stage, two 64-wide k steps of the W tile
//            [128 x 64] and the h tile [NM x 64] (128-byte swizzle) into a
//            ring of S stages;
//   warp 1   MMA issuer: 8 tcgen05.mma (K = 16 each) per stage into one of
//            two TMEM accumulators; commits free the stage, and a finished
//            tile's accumulator;
//   warp 2   allocates and frees the TMEM columns;
//   warps 4-7 epilogue: each reads its 32-lane quadrant of the finished
//            accumulator (tcgen05.ld), forms the packed (logit, full id) key
//            of every row and keeps the best per hidden row (argmax), or -
//            for top-k - passes the keys through shared memory so that lane
//            m folds hidden row m's 32 keys of the tile into its own list.
// The block's best keys then go through the same cross-block finish as the
// CUDA-core kernels.  Every mbarrier wait is bounded (about 2 s); on a
// timeout the block records DVL_ERR_TIMEOUT, stops, waits (bounded) for its
// copies and MMAs in flight and frees its TMEM before leaving.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

#include "dvl.h"
#include "dvl_device.cuh"
#include "dvl_tc.cuh"

namespace dvl {
namespace {

constexpr int kThreads = 256;
constexpr int kBM = 128;               // head rows per tile (MMA M)
constexpr int kBK = 64;                // k per stage (one 128-byte swizzle row)
constexpr int kWTile = kBM * kBK * 2;  // 16 KB
constexpr int kEpiWarp0 = 4;           // warps 4..7: TMEM lane quadrants 0..3


template <int NM, int KM>
struct TcLayout {
    static constexpr int kHTile = NM * kBK * 2;
    // 64-wide k boxes per pipeline stage and stages in the ring, measured on
    // GB300 (52,755-row head): three boxes per stage for 16 hidden-row
    // columns (1.3% faster than two), two for 32 (three leave room for too
    // few stages there: 8% slower).  Argmax has no key tile, and its shared
    // memory takes one stage more (1.2-1.9% faster): 4 x 3 boxes for 16
    // columns, 5 x 2 for 32; top-k keeps 3 x 3 and 4 x 2.
    static constexpr int kBoxes = NM == 32 ? 2 : 3;
    static constexpr int kWStage = kBoxes * kWTile;
    static constexpr int kHStage = kBoxes * kHTile;
    static constexpr int kStages = NM == 32 ? (KM == 1 ? 5 : 4) : (KM == 1 ? 4 : 3);
    static constexpr int kTmemCols = 2 * NM < 32 ? 32 : 2 * NM;
    static constexpr size_t w_off = 0;
    static constexpr size_t h_off = w_off + (size_t)kStages * kWStage;
    static constexpr size_t bar_off = h_off + (size_t)kStages * kHStage;
    // full[S], empty[S], tmem_full[2], tmem_empty[2], drain
    static constexpr size_t misc_off = bar_off + (size_t)(2 * kStages + 5) * 8;
    // tmem base, abort flag, issued, consumed
    static constexpr size_t cand_off = misc_off + 16;
    // top-k: per epilogue warp, its 32 rows' keys for every hidden row
    // [32][NM + 1] (one pad key per row spreads a column over the banks)
    static constexpr size_t keys_off = cand_off + (size_t)DVL_MAX_M * 4 * KM * 8;
    static constexpr size_t kKeyRow = NM + 1;
    static constexpr size_t bytes = keys_off + (KM > 1 ? (size_t)4 * 32 * kKeyRow * 8 : 0);
    static constexpr size_t dyn_bytes = bytes + 1024;  // room to align the base to 1 KB
};

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Bounded wait that also gives up when another role has aborted the block.
// On a timeout it raises the block's abort flag and the workspace status.
__device__ __noinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity,
                                           volatile uint32_t *abort_flag, unsigned char *ws)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity))
                return true;
        if (*abort_flag)
            return false;
        if (globaltimer_ns() - t0 > 2000000000ull) {
            *abort_flag = 1u;
            set_status(ws, 1u << DVL_ERR_TIMEOUT);
            return false;
        }
    }
}

template <int NM, int KM>
__global__ void __launch_bounds__(kThreads, 1)
    argmax_tc_kernel(const __grid_constant__ CUtensorMap tmap_w,
                     const __grid_constant__ CUtensorMap tmap_h, const ArgmaxArgs a, const int M)
{
    using L = TcLayout<NM, KM>;
    constexpr int S = L::kStages;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    unsigned char *sW = smem + L::w_off;
    unsigned char *sH = smem + L::h_off;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::bar_off);
    uint64_t *empty = full + S;
    uint64_t *tfull = empty + S;   // [2] accumulator b finished
    uint64_t *tempty = tfull + 2;  // [2] accumulator b read out
    uint64_t *drain = tempty + 2;
    // misc[0] TMEM base, [1] abort flag, [2] stages issued, [3] stages consumed
    volatile uint32_t *misc = reinterpret_cast<volatile uint32_t *>(smem + L::misc_off);
    uint64_t *s_cand = reinterpret_cast<uint64_t *>(smem + L::cand_off);  // [M][4][KM]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int KC = a.K / kBK;
    const int G = gridDim.x;
    const int r0 = (int)((long long)a.N * blockIdx.x / G);
    const int r1 = (int)((long long)a.N * (blockIdx.x + 1) / G);
    const int ntiles = (r1 - r0 + kBM - 1) / kBM;
    constexpr uint32_t idesc = tc::idesc_bf16_f32(kBM, NM);

    pdl_launch_dependents();
    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], 4);  // one arrival per epilogue warp
        }
        mbar_init(drain, 1);
        misc[1] = 0u;
        misc[2] = 0u;
        misc[3] = 0u;
        mbar_fence_init();
        tc::prefetch_tmap(&tmap_w);
        tc::prefetch_tmap(&tmap_h);
    }
    if (warp == 2)
        tc::tmem_alloc(const_cast<uint32_t *>(misc), L::kTmemCols);
    tc::fence_before_thread_sync();
    __syncthreads();
    tc::fence_after_thread_sync();
    const uint32_t tmem_base = misc[0];
    volatile uint32_t *abort_flag = misc + 1;

    if (warp == 0) {
        // ---- TMA producer ----
        // Stage i (tile i / nst, k boxes from (i % nst) * kBoxes): the W
        // boxes and the h boxes of a stage complete one barrier phase
        // together (one arrival, their bytes expected up front).  A head
        // the caller marked static fills the first S stages' W boxes before
        // the wait for the preceding kernel, their h boxes after it.
        if (lane == 0) {
            const int nst = (KC + L::kBoxes - 1) / L::kBoxes, total = ntiles * nst;
            auto boxes = [&](int i) { return min(L::kBoxes, KC - (i % nst) * L::kBoxes); };
            auto expect = [&](int i, int s) {
                mbar_arrive_expect_tx(&full[s], (uint32_t)(boxes(i) * (kWTile + L::kHTile)));
            };
            auto load_w = [&](int i, int s) {
                const int row = r0 + (i / nst) * kBM, kc = (i % nst) * L::kBoxes;
                for (int bx = 0; bx < boxes(i); ++bx)
                    tc::tma_load_2d(sW + (size_t)s * L::kWStage + bx * kWTile, &tmap_w,
                                    (kc + bx) * kBK, row, &full[s]);
            };
            auto load_h = [&](int i, int s) {
                const int kc = (i % nst) * L::kBoxes;
                for (int bx = 0; bx < boxes(i); ++bx)
                    tc::tma_load_2d(sH + (size_t)s * L::kHStage + bx * L::kHTile, &tmap_h,
                                    (kc + bx) * kBK, 0, &full[s]);
            };
            const int pre = a.head_static ? min(S, total) : 0;
            for (int i = 0; i < pre; ++i) {  // fresh barriers: no wait for the stage
                expect(i, i);
                load_w(i, i);
            }
            pdl_wait();
            for (int i = 0; i < pre; ++i) {
                load_h(i, i);
                misc[2] = i + 1;
            }
            for (int i = pre; i < total; ++i) {
                const int s = i % S;
                if (!wait_or_abort(&empty[s], ((i / S) & 1u) ^ 1u, abort_flag, a.ws))
                    break;
                expect(i, s);
                load_w(i, s);
                load_h(i, s);
                misc[2] = i + 1;
            }
        }
    } else if (warp == 1) {
        // ---- MMA issuer ----
        if (lane == 0) {
            uint32_t i = 0;
            for (int t = 0; t < ntiles; ++t) {
                const int b = t & 1;
                if (!wait_or_abort(&tempty[b], ((t >> 1) & 1) ^ 1, abort_flag, a.ws))
                    break;
                tc::fence_after_thread_sync();
                const uint32_t d = tmem_base + (uint32_t)(b * NM);
                bool ok = true;
                for (int kc = 0; kc < KC; kc += L::kBoxes, ++i) {
                    const int s = (int)(i % S);
                    if (!wait_or_abort(&full[s], (i / S) & 1u, abort_flag, a.ws)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after_thread_sync();
                    const int nb = min(L::kBoxes, KC - kc);
                    for (int bx = 0; bx < nb; ++bx) {
                        const unsigned char *wt = sW + (size_t)s * L::kWStage + bx * kWTile;
                        const unsigned char *ht = sH + (size_t)s * L::kHStage + bx * L::kHTile;
#pragma unroll
                        for (int k16 = 0; k16 < kBK / 16; ++k16)
                            tc::mma_bf16(d, tc::sw128_kmajor_desc(wt + 32 * k16),
                                         tc::sw128_kmajor_desc(ht + 32 * k16), idesc,
                                         (kc + bx) > 0 || k16 > 0);
                    }
                    tc::mma_commit(&empty[s]);  // the stage is free once these MMAs finish
                    misc[3] = i + 1;
                }
                if (!ok)
                    break;
                tc::mma_commit(&tfull[b]);
            }
            // Every MMA issued has completed before the TMEM is freed.
            tc::mma_commit(drain);
            mbar_wait_bounded(drain, 0);
        }
    } else if (warp >= kEpiWarp0) {
        // ---- epilogue: TMEM quadrant q holds rows q*32 .. q*32+31 ----
        const int q = warp - kEpiWarp0;
        uint64_t best[KM == 1 ? NM : 1];  // argmax: the best key per hidden row
#pragma unroll
        for (int m = 0; m < (KM == 1 ? NM : 1); ++m)
            best[m] = 0ull;
        TopList<KM> mine;  // top-k: lane m keeps hidden row m's list
        mine.init();
        pdl_wait();
        for (int t = 0; t < ntiles; ++t) {
            const int b = t & 1;
            const bool ok = wait_or_abort(&tfull[b], (t >> 1) & 1, abort_flag, a.ws);
            if (!__all_sync(kFull, ok))
                break;
            tc::fence_after_thread_sync();
            uint32_t v[NM];
            const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * NM);
            if constexpr (NM == 32)
                tc::tmem_ld_32x32b_x32(taddr, v);
            else
                tc::tmem_ld_32x32b_x16(taddr, v);
            tc::tmem_ld_wait();
            tc::fence_before_thread_sync();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&tempty[b]);
            const int row = r0 + t * kBM + q * 32 + lane;
            const bool in = row < r1;
            const int id = in ? (a.d2t ? __ldg(a.d2t + row) : (int)(a.id_base + row)) : 0;
            if constexpr (KM == 1) {
                if (in) {
#pragma unroll
                    for (int m = 0; m < NM; ++m) {
                        if (m < M) {
                            const uint64_t key = make_key(__uint_as_float(v[m]), id);
                            best[m] = key > best[m] ? key : best[m];
                        }
                    }
                }
            } else {
                // transpose through shared memory: each lane writes its row's
                // keys, then lane m folds hidden row m's 32 keys into its list
                uint64_t *sk = reinterpret_cast<uint64_t *>(smem + L::keys_off) +
                               (size_t)q * 32 * L::kKeyRow;
#pragma unroll
                for (int m = 0; m < NM; ++m)
                    if (m < M)
                        sk[lane * L::kKeyRow + m] = in ? make_key(__uint_as_float(v[m]), id) : 0ull;
                __syncwarp();
                if (lane < M) {
                    // most keys lose to the list's last entry: one compare each
#pragma unroll 4
                    for (int r = 0; r < 32; ++r) {
                        const uint64_t key = sk[r * L::kKeyRow + lane];
                        if (key > mine.v[KM - 1])
                            mine.insert(key);
                    }
                }
                __syncwarp();
            }
        }
        if constexpr (KM == 1) {
#pragma unroll
            for (int m = 0; m < NM; ++m) {
                if (m < M) {
                    const uint64_t k = warp_max_u64(best[m]);
                    if (lane == 0)
                        s_cand[m * 4 + q] = k;
                }
            }
        } else if (lane < M) {
#pragma unroll
            for (int i = 0; i < KM; ++i)
                s_cand[(lane * 4 + q) * KM + i] = mine.v[i];
        }
    }
    __syncthreads();
    if (*abort_flag && threadIdx.x == 0) {
        // Copies issued but never consumed must land before the block ends.
        for (uint32_t i = misc[3]; i < misc[2]; ++i)
            mbar_wait_bounded(&full[i % S], (i / S) & 1u);
    }
    tc::fence_before_thread_sync();
    __syncthreads();
    tc::fence_after_thread_sync();
    if (warp == 2)
        tc::tmem_dealloc(tmem_base, L::kTmemCols);
    block_finish<KM>(s_cand, M, 4, a);
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against the driver library).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// A 2-D bf16 tensor [rows][K] (row-major) read in boxes of box_rows x 64
// with the 128-byte swizzle; rows past the end read as zeros.
bool encode_bf16_2d(CUtensorMap *m, const void *base, int K, int rows, int box_rows)
{
    auto fn = encode_fn();
    if (!fn)
        return false;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

template <int NM, int KM>
cudaError_t launch_nm(const ArgmaxArgs &a, int M, cudaStream_t s)
{
    using L = TcLayout<NM, KM>;
    alignas(64) CUtensorMap tw, th;
    std::memset(&tw, 0, sizeof tw);
    std::memset(&th, 0, sizeof th);
    if (!encode_bf16_2d(&tw, a.w, a.K, a.N, kBM) || !encode_bf16_2d(&th, a.h, a.K, M, NM))
        return cudaErrorInvalidValue;
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess)
        return e;
    auto kern = argmax_tc_kernel<NM, KM>;
    int per_sm = 0;
    e = blocks_per_sm(reinterpret_cast<const void *>(kern), kThreads, L::dyn_bytes, &per_sm);
    if (e != cudaSuccess)
        return e;
    if (per_sm < 1)
        return cudaErrorInvalidConfiguration;
    // Few tiles per block, and rows split so each block's last tile is
    // nearly full (the tiles of a block never read far into the next's rows).
    const long long tiles = ((long long)a.N + kBM - 1) / kBM;
    long long tpb = (tiles + di.sms - 1) / di.sms;
    long long grid = ((long long)a.N + kBM * tpb - 1) / (kBM * tpb);
    if (grid > kMaxCtas)
        grid = kMaxCtas;
    if (grid < 1)
        grid = 1;
    return launch_pdl(kern, (unsigned)grid, kThreads, L::dyn_bytes, s, tw, th, a, M);
}

}  // namespace

bool tc_argmax_supported(int M, int K) { return M > 4 && M <= 32 && K % kBK == 0; }

cudaError_t launch_argmax_tc(const ArgmaxArgs &a, int M, int kmax, cudaStream_t s)
{
    if (kmax == 1)
        return M <= 16 ? launch_nm<16, 1>(a, M, s) : launch_nm<32, 1>(a, M, s);
    return M <= 16 ? launch_nm<16, 4>(a, M, s) : launch_nm<32, 4>(a, M, s);
}

}  // namespace dvl
