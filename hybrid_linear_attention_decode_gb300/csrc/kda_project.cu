// kda_project.cu -- the input projections of a KDA layer as one tcgen05 GEMM: x [T][hidden] times a packed
// weight matrix W [N][hidden] gives q, k, v, the decay logits a, the output gate z and the beta logits b, each
// written straight into the [T][H][d] layout the prefill kernels read ("A Preview of Production-Scale Kimi
// K3 Support on vLLM", section "KDA prefill and decode": the input projections and the causal convolution
// are fused around the core recurrence).  The causal convolution itself is fused into the prefill's chunk
// kernel, which reads these raw rows anyway, so the path has no separate conv pass.
//
// Design (sm_103a):
//   * persistent: one CTA of 6 warps per SM walks 128 x 256 output tiles; K in steps of 64 bf16 (one
//     128-byte swizzle atom);
//   * a 4-stage pipeline of 2-D TMA tensor loads (128B swizzle, the K-major layout the MMA descriptors
//     read), with full / empty mbarriers; warp 0 produces, warp 1 issues tcgen05.mma (M 128, N 256, K 16)
//     and commits each stage back to the producer;
//   * two 128 x 256 fp32 accumulators in tensor memory (512 columns): while the MMAs fill one, the
//     epilogue warps 2..5 (one lane quadrant, i.e. 32 token rows, each) read the other with tcgen05.ld,
//     round to bf16 and store 16-byte groups into the projection each column belongs to;
//   * tiles are rastered in groups of 16 M-tiles, so the weight tiles in flight stay in L2 while every
//     token tile of the group uses them.
// Every wait is bounded; a wait that gives up sets KDA_DEV_TIMEOUT and the tile is not stored.
#include <cuda.h>

#include <algorithm>
#include <atomic>

#include "kda_device.cuh"
#include "kda_internal.h"
#include "kda_umma.cuh"

namespace kda {
namespace proj {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4, NT = 192, GM = 16;
constexpr uint32_t A_BYTES = BM * BK * 2;
constexpr uint32_t B_BYTES = BN * BK * 2;
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
constexpr uint32_t OFF_BAR = STAGES * STAGE_BYTES;
constexpr uint32_t SMEM = OFF_BAR + 256 + 1024;  // barriers and the tensor-memory address, + alignment slack
static_assert(A_BYTES % 1024 == 0 && STAGE_BYTES % 1024 == 0, "1024-byte aligned swizzle atoms");

struct Args {
    int64_t T;
    int32_t hidden, N, ntm, ntn;
    int32_t seg_end[6];  // cumulative column ends of q, k, v, a, z, b
    int32_t seg_w[6];    // column widths (H * d, or H for b)
    uint16_t *out[6];    // destinations (z may be NULL: those columns are not stored)
    int32_t *status;
};

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int c0, int c1, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
            "r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_addr(bar))
        : "memory");
}

// Columns [n, n + 8) of one token row: a 16-byte store when they lie in one projection at an aligned
// offset, else element by element.
__device__ __forceinline__ void store8(const Args &p, int64_t row, int n, const float *v) {
    int s = 0;
    while (s < 5 && n >= p.seg_end[s]) ++s;
    const int beg = s ? p.seg_end[s - 1] : 0;
    if (n + 8 <= p.seg_end[s] && (p.seg_w[s] & 7) == 0 && ((n - beg) & 7) == 0) {
        if (p.out[s])
            *reinterpret_cast<uint4 *>(p.out[s] + row * p.seg_w[s] + (n - beg)) =
                make_uint4(umma::pack_bf16(v[0], v[1]), umma::pack_bf16(v[2], v[3]), umma::pack_bf16(v[4], v[5]),
                           umma::pack_bf16(v[6], v[7]));
        return;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const int c = n + u;
        int t = 0;
        while (t < 5 && c >= p.seg_end[t]) ++t;
        const int b0 = t ? p.seg_end[t - 1] : 0;
        if (c < p.N && p.out[t]) p.out[t][row * p.seg_w[t] + (c - b0)] = f2bf(v[u]);
    }
}

// Tile `t` of the raster: groups of GM M-tiles, M fastest inside a group.
__device__ __forceinline__ void tile_coords(const Args &p, int t, int &tm, int &tn) {
    const int per_group = GM * p.ntn;
    const int g = t / per_group, rem = t - g * per_group;
    const int gm0 = g * GM, gsz = min(GM, p.ntm - gm0);
    tm = gm0 + rem % gsz;
    tn = rem / gsz;
}

__global__ void __launch_bounds__(NT, 1)
    kda_project_kernel(const Args p, const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + OFF_BAR);  // [STAGES] stage loaded
    uint64_t *empty = full + STAGES;                               // [STAGES] stage consumed by the MMAs
    uint64_t *acc_full = empty + STAGES;                           // [2] accumulator complete
    uint64_t *acc_empty = acc_full + 2;                            // [2] accumulator read by the epilogue
    uint32_t *tmem_s = reinterpret_cast<uint32_t *>(acc_empty + 2);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int ntiles = p.ntm * p.ntn;
    const int nk = (p.hidden + BK - 1) / BK;

    if (warp == 0) umma::alloc(tmem_s, 2 * BN);
    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
        }
        for (int a2 = 0; a2 < 2; ++a2) {
            mbar_init(acc_full + a2, 1);
            mbar_init(acc_empty + a2, 4);  // one arrival per epilogue warp
        }
        fence_mbar_init();
    }
    umma::fence_before();
    __syncthreads();
    umma::fence_after();
    const uint32_t tmem = *tmem_s;
    bool ok = true;
    int kg = 0;  // producer: K steps whose loads were issued; MMA issuer: K steps whose MMAs were issued

    if (warp == 0) {
        if (lane == 0) {  // producer: TMA loads of the x and W tiles of every K step of every tile
            // K step kg (counted over all tiles) uses stage kg % STAGES for the (kg / STAGES)-th time
            for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
                int tm, tn;
                tile_coords(p, t, tm, tn);
                for (int kb = 0; kb < nk; ++kb, ++kg) {
                    const int s = kg % STAGES;
                    if (kg >= STAGES && !mbar_wait(empty + s, (uint32_t)(kg / STAGES - 1) & 1u)) {
                        ok = false;
                        break;
                    }
                    uint8_t *sa = sm + s * STAGE_BYTES;
                    mbar_arrive_expect_tx(full + s, STAGE_BYTES);
                    tma_load_2d(sa, &tm_x, kb * BK, tm * BM, full + s);
                    tma_load_2d(sa + A_BYTES, &tm_w, kb * BK, tn * BN, full + s);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {  // MMA issuer: accumulator i % 2 for the i-th tile of this CTA
            const uint32_t id = umma::idesc(umma::kBF16, BM, BN);
            int i = 0;
            for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x, ++i) {
                const int a2 = i & 1;
                if (i >= 2 && !mbar_wait(acc_empty + a2, (uint32_t)(i / 2 - 1) & 1u)) {
                    ok = false;
                    break;
                }
                umma::fence_after();
                const uint32_t acc = tmem + (uint32_t)(a2 * BN);
                for (int kb = 0; kb < nk; ++kb, ++kg) {
                    const int s = kg % STAGES;
                    if (!mbar_wait(full + s, (uint32_t)(kg / STAGES) & 1u)) {
                        ok = false;
                        break;
                    }
                    umma::fence_after();
                    const uint8_t *sa = sm + s * STAGE_BYTES;
#pragma unroll
                    for (int ks = 0; ks < BK / 16; ++ks)
                        umma::mma_bf16(acc, umma::sdesc_k(sa, BM, ks), umma::sdesc_k(sa + A_BYTES, BN, ks), id,
                                       kb > 0 || ks > 0);
                    umma::commit(empty + s);  // the stage is free once these MMAs have read it
                }
                if (ok) umma::commit(acc_full + a2);
            }
        }
    } else if (warp < 6) {  // epilogue warps 2..5: tensor-memory lane quadrant warp % 4 = rows of the tile
        const int quad = warp & 3;
        int i = 0;
        for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++i) {
            const int a2 = i & 1;
            if (!__all_sync(0xffffffffu, mbar_wait(acc_full + a2, (uint32_t)(i / 2) & 1u))) {
                ok = false;
                break;
            }
            umma::fence_after();
            int tm, tn;
            tile_coords(p, t, tm, tn);
            const int64_t row = (int64_t)tm * BM + quad * 32 + lane;
            const uint32_t acc = tmem + (uint32_t)(a2 * BN) + ((uint32_t)(32 * quad) << 16);
            for (int cg = 0; cg < BN / 32; ++cg) {
                float v[32];
                umma::ld32(acc + 32 * cg, v);
                const int n0 = tn * BN + 32 * cg;
                if (row < p.T && n0 < p.N) {
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (n0 + 8 * j < p.N) store8(p, row, n0 + 8 * j, v + 8 * j);
                }
            }
            umma::fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_expect_tx(acc_empty + a2, 0);  // this quadrant of the accumulator is read
        }
    }
    if (!ok && lane == 0) set_status(p.status, KDA_DEV_TIMEOUT);
    // After a timed-out wait anywhere in the CTA, loads may still be landing in its shared memory and MMAs
    // may still be reading it and writing the accumulators: the producer waits for its last STAGES loads and
    // the MMA issuer for the commit of its last MMAs (which covers every earlier one), briefly and bounded,
    // before the tensor memory is freed and the CTA exits.
    if (__syncthreads_or(!ok) && lane == 0 && warp < 2) {
        constexpr uint64_t kDrainNs = 10000000ull;
        if (warp == 0) {
            for (int j = kg > STAGES ? kg - STAGES : 0; j < kg; ++j)
                mbar_wait(full + j % STAGES, (uint32_t)(j / STAGES) & 1u, kDrainNs);
        } else if (kg > 0) {
            mbar_wait(empty + (kg - 1) % STAGES, (uint32_t)((kg - 1) / STAGES) & 1u, kDrainNs);
        }
    }
    umma::fence_before();
    __syncthreads();
    if (warp == 0) umma::dealloc(tmem, 2 * BN);
}

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encoder() {
    static std::atomic<EncodeTiledFn> cached{nullptr};
    EncodeTiledFn f = cached.load(std::memory_order_acquire);
    if (f) return f;
    void *fp = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fp, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fp)
        return nullptr;
    f = reinterpret_cast<EncodeTiledFn>(fp);
    cached.store(f, std::memory_order_release);
    return f;
}

// A row-major [rows][K] bf16 matrix as a 2-D map with 64 x box_rows boxes in the 128-byte swizzle.
static bool kmajor_map(EncodeTiledFn enc, CUtensorMap *m, const void *base, int64_t K, int64_t rows, int box_rows) {
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1u, 1u};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace proj

int launch_project(const ProjectArgs &a, cudaStream_t st) {
    using namespace proj;
    static int attr_done[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return launch_result("project: cudaGetDevice");
    if (!attr_done[dev]) {
        if (cudaFuncSetAttribute(kda_project_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM) != cudaSuccess)
            return launch_result("project: cudaFuncSetAttribute");
        attr_done[dev] = 1;
    }
    const EncodeTiledFn enc = encoder();
    if (!enc) return fail(KDA_ERR_CUDA, "project: cuTensorMapEncodeTiled is not available");
    Args p;
    p.T = a.T;
    p.hidden = a.hidden;
    const int H = a.H;
    const int w[6] = {H * a.dk, H * a.dk, H * a.dv, H * a.dk, H * a.dv, H};
    int acc = 0;
    for (int s = 0; s < 6; ++s) {
        acc += w[s];
        p.seg_end[s] = acc;
        p.seg_w[s] = w[s];
    }
    p.N = acc;
    p.out[0] = a.q; p.out[1] = a.k; p.out[2] = a.v; p.out[3] = a.a; p.out[4] = a.z; p.out[5] = a.b;
    p.status = a.status;
    const int64_t ntm = (a.T + BM - 1) / BM, ntn = (p.N + BN - 1) / BN;
    if (ntm * ntn > 0x7fffffffLL) return fail(KDA_ERR_INVALID_ARG, "project: too many tiles");
    p.ntm = (int32_t)ntm;
    p.ntn = (int32_t)ntn;
    CUtensorMap tx, tw;
    if (!kmajor_map(enc, &tx, a.x, a.hidden, a.T, BM) || !kmajor_map(enc, &tw, a.w, a.hidden, p.N, BN))
        return fail(KDA_ERR_CUDA, "project: tensor map encoding failed");
    const unsigned grid = (unsigned)std::min<int64_t>(ntm * ntn, current_device_sms());  // persistent: one per SM
    kda_project_kernel<<<grid, NT, SMEM, st>>>(p, tx, tw);
    return launch_result("kda_project_kernel launch");
}

}  // namespace kda
