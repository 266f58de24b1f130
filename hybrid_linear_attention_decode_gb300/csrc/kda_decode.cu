// kda_decode.cu -- fused KDA decode step for sm_103a.
//
// One decode token per request: causal conv + SiLU, q/k L2-norm, sigmoid gates, gated delta-rule state
// update, readout and gated RMSNorm in a single launch ("A Preview of Production-Scale Kimi K3
// Support on vLLM", section "KDA prefill and decode"; "vLLM Kimi K3 Support", section "Fused Kernels
// and Metadata Optimization").
//
// The step is a stream over fp32 states (64 KiB per request and head at dk = dv = 128): each state is
// read once and written once.  Design:
//   * persistent CTAs (two per SM at dk = dv = 128), each walking work items (request, head) with a
//     stride of gridDim.x, heads fastest so that neighbouring CTAs stream neighbouring 64 KiB tiles of
//     one slot;
//   * every input of an item -- the state in NST stages, the raw conv window, q, k, v, a, z -- arrives
//     by 1-D bulk TMA copies into one of NBUF shared-memory buffers, completion counted on mbarriers;
//     the state moves to registers in the first pass, after which the buffer is handed to the copies
//     of a later item, so loads overlap the rest of the item and the other CTA's work;
//   * one pass over S' = Diag(alpha) S reduces k^T S' and q^T S' together (o = S'^T q + beta (k.q) u
//     with u = v - S'^T k), a second pass writes S' + beta k u^T with 128-bit coalesced stores;
//   * conv, norms and gates use warp reductions in a fixed order, so the kernel is deterministic.
#include "kda_device.cuh"
#include "kda_internal.h"

namespace kda {

// Resident CTAs per SM targeted for a bf16 pool at dk = dv = 128 (the register budget, 64 per thread,
// follows from it).  Swept on the decode workload: 4 x 1 buffer 27.8 us, 3 x 1 29.2, 2 x 1 34.2, 2 x 2 35.5,
// 3 x 2 35.4 (us per step).
#ifndef KDA_DECODE_BF16_CTAS
#define KDA_DECODE_BF16_CTAS 4
#endif
#ifndef KDA_DECODE_NBUF_BF16
#define KDA_DECODE_NBUF_BF16 1
#endif

template <int DK, int DV, int NBUF, bool SBF>
struct DecodeShape {
    static constexpr int ES = SBF ? 2 : 4;    // bytes per stored state element (bf16 or fp32 pool)
    static constexpr int W = 4;
    static constexpr int CC = 2 * DK + DV;
    static constexpr int NT = (DK * DV >= 4096) ? 256 : 64;
    static constexpr int LPR = DV / 4;        // threads per state row (one float4 each)
    static constexpr int RPP = NT / LPR;      // rows covered by the block at once
    static constexpr int RPT = DK / RPP;      // rows per thread
    static constexpr int NST = (DK >= 128) ? 4 : 1;
    static constexpr int M_ST = RPT / NST;    // rows per thread per stage
    static constexpr int CPT = (CC + NT - 1) / NT;  // conv channels per thread
    static constexpr uint32_t S_BYTES = DK * DV * ES;
    static constexpr uint32_t ST_BYTES = S_BYTES / NST;
    static constexpr uint32_t CONV_BYTES = (W - 1) * CC * 2;
    static constexpr uint32_t OFF_CONV = S_BYTES;
    static constexpr uint32_t OFF_Q = OFF_CONV + CONV_BYTES;
    static constexpr uint32_t OFF_K = OFF_Q + DK * 2;
    static constexpr uint32_t OFF_V = OFF_K + DK * 2;
    static constexpr uint32_t OFF_A = OFF_V + DV * 2;
    static constexpr uint32_t OFF_Z = OFF_A + DK * 2;
    static constexpr uint32_t BUF_BYTES = (OFF_Z + DV * 2 + 127) / 128 * 128;
    static constexpr int NF = 2 * RPP * DV + CC + 4 * DK + 3 * DV;  // float scratch
    static constexpr uint32_t OFF_F = NBUF * BUF_BYTES;
    static constexpr uint32_t OFF_BAR = (OFF_F + NF * 4 + 15) / 16 * 16;
    static constexpr uint32_t SMEM = OFF_BAR + NBUF * (1 + NST) * 8;
    static constexpr int MIN_BLOCKS = (DK * DV >= 4096) ? (SBF ? KDA_DECODE_BF16_CTAS : (NBUF == 1 ? 2 : 1)) : 1;

    static_assert(LPR <= 32 && 32 % LPR == 0, "row mapping");
    static_assert(DV <= NT, "one output channel per thread in the epilogue");
    static_assert(RPP * RPT == DK && RPT % NST == 0, "row split");
    static_assert(CONV_BYTES % 16 == 0 && (DK * 2) % 16 == 0 && (DV * 2) % 16 == 0, "bulk copy sizes");
    static_assert(OFF_CONV % 16 == 0 && OFF_Q % 16 == 0 && OFF_V % 16 == 0 && OFF_A % 16 == 0, "align");
};

template <int DK, int DV, int NBUF, bool SBF>
__global__ void __launch_bounds__(DecodeShape<DK, DV, NBUF, SBF>::NT, DecodeShape<DK, DV, NBUF, SBF>::MIN_BLOCKS)
    kda_decode_kernel(const DecodeArgs args) {
    using C = DecodeShape<DK, DV, NBUF, SBF>;
    constexpr int NT = C::NT, CC = C::CC, NST = C::NST, RPP = C::RPP, LPR = C::LPR, RPT = C::RPT;
    extern __shared__ __align__(128) uint8_t smem[];
    float *red_k = reinterpret_cast<float *>(smem + C::OFF_F);  // [RPP][DV]
    float *red_q = red_k + RPP * DV;                              // [RPP][DV]
    float *xs = red_q + RPP * DV;                                 // [CC] conv outputs
    float *kh = xs + CC;                                          // [DK] k^
    float *ka = kh + DK;                                          // [DK] alpha * k^
    float *qa = ka + DK;                                          // [DK] alpha * q^
    float *al = qa + DK;                                          // [DK] alpha
    float *bu = al + DK;                                          // [DV] beta * u
    float *os = bu + DV;                                          // [DV] o
    float *nw = os + DV;                                          // [DV] RMSNorm weight
    uint64_t *bar_in = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);  // [NBUF]
    uint64_t *bar_S = bar_in + NBUF;                                      // [NBUF][NST]

    const int tid = threadIdx.x;
    const int H = args.H;
    const int nitems = args.n * H;
    const int64_t ns = args.num_slots;

    if (tid == 0) {
        for (int i = 0; i < NBUF * (1 + NST); ++i) mbar_init(&bar_in[i], 1);
        fence_mbar_init();
    }
    for (int j = tid; j < DV; j += NT) nw[j] = __ldg(args.norm_w + j);
    __syncthreads();

    // Thread 0: start every copy of `item` into buffer `buf`.  Each barrier of the buffer is arrived
    // on exactly once per use (with 0 expected bytes when there is nothing to copy), so phase parity
    // always equals the buffer's use count.
    auto issue = [&](int buf, int item) {
        if (item >= nitems) return;
        const int n = item / H, h = item - (item / H) * H;
        const int src = args.src[n], dst = args.dst[n];
        const bool ok = src >= -1 && src < ns && dst >= 0 && dst < ns;
        uint8_t *bp = smem + (size_t)buf * C::BUF_BYTES;
        uint64_t *bi = &bar_in[buf];
        uint64_t *bs = &bar_S[buf * NST];
        if (!ok) {
            mbar_arrive_expect_tx(bi, 0);
            for (int s = 0; s < NST; ++s) mbar_arrive_expect_tx(&bs[s], 0);
            return;
        }
        const size_t th = (size_t)n * H + h;
        const uint32_t bytes = 3 * DK * 2 + DV * 2 + (args.z ? DV * 2 : 0) + (src >= 0 ? C::CONV_BYTES : 0);
        mbar_arrive_expect_tx(bi, bytes);
        bulk_g2s(bp + C::OFF_Q, args.q + th * DK, DK * 2, bi);
        bulk_g2s(bp + C::OFF_K, args.k + th * DK, DK * 2, bi);
        bulk_g2s(bp + C::OFF_V, args.v + th * DV, DV * 2, bi);
        bulk_g2s(bp + C::OFF_A, args.a + th * DK, DK * 2, bi);
        if (args.z) bulk_g2s(bp + C::OFF_Z, args.z + th * DV, DV * 2, bi);
        if (src >= 0) {
            const size_t sh = (size_t)src * H + h;
            bulk_g2s(bp + C::OFF_CONV, args.conv + sh * (C::W - 1) * CC, C::CONV_BYTES, bi);
            const uint8_t *gS = reinterpret_cast<const uint8_t *>(args.S) + sh * C::S_BYTES;
            for (int s = 0; s < NST; ++s) {
                mbar_arrive_expect_tx(&bs[s], C::ST_BYTES);
                bulk_g2s(bp + s * C::ST_BYTES, gS + (size_t)s * C::ST_BYTES, C::ST_BYTES, &bs[s]);
            }
        } else {
            for (int s = 0; s < NST; ++s) mbar_arrive_expect_tx(&bs[s], 0);
        }
    };

    if (tid == 0)
        for (int b = 0; b < NBUF; ++b) issue(b, blockIdx.x + b * gridDim.x);

    // Thread 0, on the exit after a timed-out wait in iteration `it`: copies issued for iterations it ..
    // it + NBUF - 1 (one per buffer, the last phase armed on its barriers) may still be landing in this CTA's
    // shared memory; wait for each, briefly and bounded, before the CTA exits.
    auto drain = [&](int it) {
        constexpr uint64_t kDrainNs = 10000000ull;
        for (int j = it; j < it + NBUF && blockIdx.x + j * (int)gridDim.x < nitems; ++j) {
            const int b = j % NBUF;
            const uint32_t p = (uint32_t)(j / NBUF) & 1u;
            mbar_wait(&bar_in[b], p, kDrainNs);
            for (int s = 0; s < NST; ++s) mbar_wait(&bar_S[b * NST + s], p, kDrainNs);
        }
    };

    const int g = tid / LPR, cg = tid - (tid / LPR) * LPR;
    for (int it = 0;; ++it) {
        const int item = blockIdx.x + it * gridDim.x;
        if (item >= nitems) break;
        const int buf = it % NBUF;
        const uint32_t par = (uint32_t)(it / NBUF) & 1u;
        const int n = item / H, h = item - (item / H) * H;
        const int src = __ldg(args.src + n), dst = __ldg(args.dst + n);
        const bool ok = src >= -1 && src < ns && dst >= 0 && dst < ns;
        const size_t th = (size_t)n * H + h;
        uint8_t *bp = smem + (size_t)buf * C::BUF_BYTES;
        const float *Ss = reinterpret_cast<const float *>(bp);
        const uint16_t *cs = reinterpret_cast<const uint16_t *>(bp + C::OFF_CONV);
        const uint16_t *q_s = reinterpret_cast<const uint16_t *>(bp + C::OFF_Q);
        const uint16_t *a_s = reinterpret_cast<const uint16_t *>(bp + C::OFF_A);
        const uint16_t *z_s = reinterpret_cast<const uint16_t *>(bp + C::OFF_Z);

        // global loads that do not depend on the copies: issued before the wait
        float4 wc[C::CPT];
#pragma unroll
        for (int u = 0; u < C::CPT; ++u) {
            const int c = tid + u * NT;
            if (c < CC) wc[u] = __ldg(reinterpret_cast<const float4 *>(args.conv_w + ((size_t)h * CC + c) * 4));
        }
        const float beta = ok ? sigmoidf_(bf2f(__ldg(args.b + th))) : 0.f;

        bool fail = !mbar_wait(&bar_in[buf], par);
        if (__syncthreads_or(fail)) {
            if (tid == 0) {
                set_status(args.status, KDA_DEV_TIMEOUT);
                drain(it);
            }
            return;
        }
        if (!ok) {
            for (int j = tid; j < DV; j += NT) args.y[th * DV + j] = 0;
            if (tid == 0) set_status(args.status, KDA_DEV_BAD_SLOT);
            __syncthreads();  // every read of this buffer is done
            if (tid == 0) {
                fence_proxy_async_smem();
                issue(buf, item + NBUF * gridDim.x);
            }
            continue;
        }
        // ---- causal conv (+ SiLU) over the q | k | v channels; the new raw window goes to dst ----
        uint16_t *cd = args.conv + ((size_t)dst * H + h) * (C::W - 1) * CC;
#pragma unroll
        for (int u = 0; u < C::CPT; ++u) {
            const int c = tid + u * NT;
            if (c >= CC) break;
            const uint16_t xr = q_s[c];  // q, k, v are contiguous in the buffer
            uint16_t w0 = 0, w1 = 0, w2 = 0;
            if (src >= 0) {
                w0 = cs[c];
                w1 = cs[CC + c];
                w2 = cs[2 * CC + c];
            }
            const float4 w = wc[u];
            float acc = w.w * bf2f(xr);
            acc = fmaf(w.x, bf2f(w0), acc);
            acc = fmaf(w.y, bf2f(w1), acc);
            acc = fmaf(w.z, bf2f(w2), acc);
            if (args.silu) acc = acc / (1.0f + __expf(-acc));
            xs[c] = acc;
            cd[c] = w1;
            cd[CC + c] = w2;
            cd[2 * CC + c] = xr;
        }
        float zg = 1.f;
        if (args.z && tid < DV) zg = sigmoidf_(bf2f(z_s[tid]));
        __syncthreads();
        // every warp reduces |q|^2, |k|^2 and q.k itself (no extra block barrier)
        const float nq = warp_dot_array(xs, xs, DK);
        const float nk = warp_dot_array(xs + DK, xs + DK, DK);
        const float qk = warp_dot_array(xs, xs + DK, DK);
        const float rq = rsqrtf(nq + args.l2_eps), rk = rsqrtf(nk + args.l2_eps);
        const float kq = qk * rq * rk;
        for (int i = tid; i < DK; i += NT) {
            const float alpha = sigmoidf_(bf2f(a_s[i]));
            const float k_ = xs[DK + i] * rk;
            kh[i] = k_;
            al[i] = alpha;
            ka[i] = alpha * k_;
            qa[i] = alpha * (xs[i] * rq);
        }
        __syncthreads();

        // ---- pass 1: the state into registers; column sums of k^T S' and q^T S' ----
        float4 sr[SBF ? 1 : RPT];   // fp32 pool: the state slice in registers
        uint2 sh[SBF ? RPT : 1];    // bf16 pool: the same slice as packed bf16 pairs
        float4 accK = make_float4(0.f, 0.f, 0.f, 0.f), accQ = accK;
        bool sfail = false;
        if (src >= 0) {
#pragma unroll
            for (int s = 0; s < NST; ++s) {
                sfail |= !mbar_wait(&bar_S[buf * NST + s], par);
#pragma unroll
                for (int m = 0; m < C::M_ST; ++m) {
                    const int mm = s * C::M_ST + m;
                    const int row = g + mm * RPP;
                    float4 x;
                    if (SBF) {
                        const uint2 hb = *reinterpret_cast<const uint2 *>(bp + (row * DV + cg * 4) * 2);
                        sh[mm] = hb;
                        x = make_float4(bf2f((uint16_t)(hb.x & 0xffff)), bf2f((uint16_t)(hb.x >> 16)),
                                        bf2f((uint16_t)(hb.y & 0xffff)), bf2f((uint16_t)(hb.y >> 16)));
                    } else {
                        x = *reinterpret_cast<const float4 *>(Ss + row * DV + cg * 4);
                        sr[mm] = x;
                    }
                    const float kk = ka[row], qq = qa[row];
                    accK.x = fmaf(kk, x.x, accK.x); accK.y = fmaf(kk, x.y, accK.y);
                    accK.z = fmaf(kk, x.z, accK.z); accK.w = fmaf(kk, x.w, accK.w);
                    accQ.x = fmaf(qq, x.x, accQ.x); accQ.y = fmaf(qq, x.y, accQ.y);
                    accQ.z = fmaf(qq, x.z, accQ.z); accQ.w = fmaf(qq, x.w, accQ.w);
                }
            }
        } else {
#pragma unroll
            for (int mm = 0; mm < RPT; ++mm) {
                if (SBF) sh[mm] = make_uint2(0u, 0u);
                else sr[mm] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        *reinterpret_cast<float4 *>(red_k + g * DV + cg * 4) = accK;
        *reinterpret_cast<float4 *>(red_q + g * DV + cg * 4) = accQ;
        if (__syncthreads_or(sfail)) {
            if (tid == 0) {
                set_status(args.status, KDA_DEV_TIMEOUT);
                drain(it);
            }
            return;
        }
        // the buffer is no longer read: start the copies of a later item into it
        if (tid == 0) {
            fence_proxy_async_smem();
            issue(buf, item + NBUF * gridDim.x);
        }
        for (int j = tid; j < DV; j += NT) {
            float kS = 0.f, qS = 0.f;
#pragma unroll
            for (int r = 0; r < RPP; ++r) {
                kS += red_k[r * DV + j];
                qS += red_q[r * DV + j];
            }
            const float u = xs[2 * DK + j] - kS;
            os[j] = args.scale * fmaf(beta * kq, u, qS);
            bu[j] = beta * u;
        }
        __syncthreads();
        const float ss = warp_dot_array(os, os, DV);
        const float rr = rsqrtf(ss * (1.0f / DV) + args.rms_eps);
        for (int j = tid; j < DV; j += NT) args.y[th * DV + j] = f2bf(os[j] * rr * nw[j] * zg);
        // ---- pass 2: S_new = Diag(alpha) S + k^ (beta u)^T from registers, 128-bit stores ----
        uint8_t *Sd = reinterpret_cast<uint8_t *>(args.S) + ((size_t)dst * H + h) * C::S_BYTES;
        const float4 b4 = *reinterpret_cast<const float4 *>(bu + cg * 4);
#pragma unroll
        for (int mm = 0; mm < RPT; ++mm) {
            const int row = g + mm * RPP;
            const float aa = al[row], kk = kh[row];
            float4 x;
            if (SBF) {
                const uint2 hb = sh[mm];
                x = make_float4(bf2f((uint16_t)(hb.x & 0xffff)), bf2f((uint16_t)(hb.x >> 16)),
                                bf2f((uint16_t)(hb.y & 0xffff)), bf2f((uint16_t)(hb.y >> 16)));
            } else {
                x = sr[mm];
            }
            float4 o4;
            o4.x = fmaf(kk, b4.x, aa * x.x);
            o4.y = fmaf(kk, b4.y, aa * x.y);
            o4.z = fmaf(kk, b4.z, aa * x.z);
            o4.w = fmaf(kk, b4.w, aa * x.w);
            if (SBF) {
                *reinterpret_cast<uint2 *>(Sd + (row * DV + cg * 4) * 2) =
                    make_uint2((uint32_t)f2bf(o4.x) | ((uint32_t)f2bf(o4.y) << 16),
                               (uint32_t)f2bf(o4.z) | ((uint32_t)f2bf(o4.w) << 16));
            } else {
                *reinterpret_cast<float4 *>(Sd + (row * DV + cg * 4) * 4) = o4;
            }
        }
    }
}

template <int DK, int DV, int NBUF, bool SBF>
static int launch_decode_t(const DecodeArgs &a, cudaStream_t st) {
    using C = DecodeShape<DK, DV, NBUF, SBF>;
    auto kern = kda_decode_kernel<DK, DV, NBUF, SBF>;
    static int occ_cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return launch_result("decode: cudaGetDevice");
    if (occ_cache[dev] == 0) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
            return launch_result("decode: cudaFuncSetAttribute");
        int occ = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, C::NT, C::SMEM) != cudaSuccess || occ < 1)
            return fail(KDA_ERR_CUDA, "decode: the kernel cannot be resident on this device");
        occ_cache[dev] = occ;
    }
    const int items = a.n * a.H;
    const int cap = current_device_sms() * occ_cache[dev];
    const int grid = items < cap ? items : cap;
    kern<<<grid, C::NT, C::SMEM, st>>>(a);
    return launch_result("kda_decode_kernel launch");
}

bool decode_supported(int dk, int dv, int W) {
    if (W != 4) return false;
    return (dk == 16 && dv == 16) || (dk == 32 && dv == 16) || (dk == 16 && dv == 32) || (dk == 64 && dv == 64) ||
           (dk == 128 && dv == 128);
}

// Item buffers per CTA at dk = dv = 128: 1 buffer runs two CTAs per SM, 2 or 3 buffers one CTA per SM.
#ifndef KDA_DECODE_NBUF_128
#define KDA_DECODE_NBUF_128 1
#endif

template <int DK, int DV, int NBUF_F32, int NBUF_BF16>
static int launch_decode_dt(const DecodeArgs &a, cudaStream_t st) {
    return a.state_bf16 ? launch_decode_t<DK, DV, NBUF_BF16, true>(a, st) : launch_decode_t<DK, DV, NBUF_F32, false>(a, st);
}

int launch_decode(const DecodeArgs &a, int dk, int dv, cudaStream_t st) {
    if (dk == 128 && dv == 128) return launch_decode_dt<128, 128, KDA_DECODE_NBUF_128, KDA_DECODE_NBUF_BF16>(a, st);
    if (dk == 64 && dv == 64) return launch_decode_dt<64, 64, 2, 2>(a, st);
    if (dk == 16 && dv == 16) return launch_decode_dt<16, 16, 2, 2>(a, st);
    if (dk == 32 && dv == 16) return launch_decode_dt<32, 16, 2, 2>(a, st);
    if (dk == 16 && dv == 32) return launch_decode_dt<16, 32, 2, 2>(a, st);
    return KDA_ERR_UNSUPPORTED_SHAPE;
}

}  // namespace kda
