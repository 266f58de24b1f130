// kda_decode_multi.cu -- L consecutive decode tokens per request in one launch, with the state after every
// position kept on request (speculative verification: the draft tokens of a request are checked in one
// pass, and the state at the last accepted position must survive the rejection of the rest).
//
// Pages: "vLLM Kimi K3 Support", section "Speculative Decoding with DSpark" (several tokens accepted per
// step); "moonshotai/Kimi-K3" recipe (num_speculative_tokens 4); "A Preview of Production-Scale Kimi K3
// Support on vLLM", section "KDA prefill and decode" (the fused decode step this repeats L times).  The pages
// do not say how a recurrent state is rolled back; the reading here is per-position retention: the state (and
// conv window) after token j of request r goes to dst_slots[r * L + j] when that entry is not -1.
//
// Design (per (request, head) item, persistent CTAs like the single-token kernel):
//   * the state arrives once by 1-D bulk TMA (NST stages), moves to registers in the first pass of token 0
//     and stays there, in fp32, for all L tokens; its buffer is then handed to the next item;
//   * the conv window and the L tokens' q|k|v, a, z rows arrive by bulk copies into one of two input
//     buffers (the other holds the next item's);
//   * per token: conv + SiLU with the window in registers, norms, gates, one pass over the register state
//     for k^T S' and q^T S', readout + gated RMSNorm, update S <- Diag(alpha) S + k^ (beta u)^T in registers,
//     and, if that position is kept, 128-bit stores of S (rounded to bf16 for a bf16 pool) and the window.
#include "kda_device.cuh"
#include "kda_internal.h"

namespace kda {

template <int DK, int DV, bool SBF>
struct MultiShape {
    static constexpr int ES = SBF ? 2 : 4;
    static constexpr int W = 4;
    static constexpr int CC = 2 * DK + DV;
    static constexpr int NT = (DK * DV >= 4096) ? 256 : 64;
    static constexpr int LPR = DV / 4;
    static constexpr int RPP = NT / LPR;
    static constexpr int RPT = DK / RPP;
    static constexpr int NST = (DK >= 128) ? 4 : 1;
    static constexpr int M_ST = RPT / NST;
    static constexpr int CPT = (CC + NT - 1) / NT;
    static constexpr uint32_t S_BYTES = DK * DV * ES;
    static constexpr uint32_t ST_BYTES = S_BYTES / NST;
    static constexpr uint32_t CONV_BYTES = (W - 1) * CC * 2;
    // one token in an input buffer: q | k | v (contiguous, the conv channels), then a, then z
    static constexpr uint32_t T_A = CC * 2;
    static constexpr uint32_t T_Z = T_A + DK * 2;
    static constexpr uint32_t TOK_BYTES = T_Z + DV * 2;
    static constexpr uint32_t IN_BYTES = (CONV_BYTES + KDA_DECODE_MULTI_MAX_L * TOK_BYTES + 127) / 128 * 128;
    static constexpr uint32_t OFF_IN = (S_BYTES + 127) / 128 * 128;
    static constexpr int NF = 2 * RPP * DV + CC + 4 * DK + 3 * DV;
    static constexpr uint32_t OFF_F = OFF_IN + 2 * IN_BYTES;
    static constexpr uint32_t OFF_BAR = (OFF_F + NF * 4 + 15) / 16 * 16;
    static constexpr uint32_t SMEM = OFF_BAR + (2 + NST) * 8;
    static constexpr int MIN_BLOCKS = (DK * DV >= 4096) ? 2 : 1;

    static_assert(LPR <= 32 && 32 % LPR == 0, "row mapping");
    static_assert(DV <= NT, "one output channel per thread in the epilogue");
    static_assert(RPP * RPT == DK && RPT % NST == 0, "row split");
    static_assert(CONV_BYTES % 16 == 0 && TOK_BYTES % 16 == 0 && T_A % 16 == 0 && T_Z % 16 == 0, "bulk sizes");
    static_assert(ST_BYTES % 16 == 0 && OFF_IN % 128 == 0 && IN_BYTES % 128 == 0, "align");
};

template <int DK, int DV, bool SBF>
__global__ void __launch_bounds__(MultiShape<DK, DV, SBF>::NT, MultiShape<DK, DV, SBF>::MIN_BLOCKS)
    kda_decode_multi_kernel(const DecodeArgs args, const int L) {
    using C = MultiShape<DK, DV, SBF>;
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
    uint64_t *bar_in = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);  // [2] input buffers
    uint64_t *bar_S = bar_in + 2;                                         // [NST] the state buffer

    const int tid = threadIdx.x;
    const int H = args.H;
    const int nitems = args.n * H;
    const int64_t ns = args.num_slots;

    if (tid == 0) {
        for (int i = 0; i < 2 + NST; ++i) mbar_init(&bar_in[i], 1);
        fence_mbar_init();
    }
    for (int j = tid; j < DV; j += NT) nw[j] = __ldg(args.norm_w + j);
    __syncthreads();

    // Slot indices of request n are valid: src in [-1, ns), every kept-position slot in [-1, ns).
    auto request_ok = [&](int n) {
        const int src = args.src[n];
        bool ok = src >= -1 && src < ns;
        for (int j = 0; j < L; ++j) {
            const int d = args.dst[(size_t)n * L + j];
            ok = ok && d >= -1 && d < ns;
        }
        return ok;
    };
    // Thread 0: the conv window and the L tokens of `item` into input buffer ib, and its state into the
    // state buffer.  Every barrier is arrived on exactly once per use (0 bytes when nothing is copied), so
    // bar_in[ib]'s parity is its use count and bar_S's the item count of this CTA.
    auto issue = [&](int ib, int item) {
        if (item >= nitems) return;
        const int n = item / H, h = item - (item / H) * H;
        uint8_t *ip = smem + C::OFF_IN + (size_t)ib * C::IN_BYTES;
        uint64_t *bi = &bar_in[ib];
        if (!request_ok(n)) {
            mbar_arrive_expect_tx(bi, 0);
            for (int s = 0; s < NST; ++s) mbar_arrive_expect_tx(&bar_S[s], 0);
            return;
        }
        const int src = args.src[n];
        const uint32_t tok = 3 * DK * 2 + DV * 2 + (args.z ? DV * 2 : 0);
        mbar_arrive_expect_tx(bi, (uint32_t)L * tok + (src >= 0 ? C::CONV_BYTES : 0));
        for (int j = 0; j < L; ++j) {
            const size_t th = ((size_t)n * L + j) * H + h;
            uint8_t *tp = ip + C::CONV_BYTES + (size_t)j * C::TOK_BYTES;
            bulk_g2s(tp, args.q + th * DK, DK * 2, bi);
            bulk_g2s(tp + DK * 2, args.k + th * DK, DK * 2, bi);
            bulk_g2s(tp + 2 * DK * 2, args.v + th * DV, DV * 2, bi);
            bulk_g2s(tp + C::T_A, args.a + th * DK, DK * 2, bi);
            if (args.z) bulk_g2s(tp + C::T_Z, args.z + th * DV, DV * 2, bi);
        }
        if (src >= 0) {
            const size_t sh = (size_t)src * H + h;
            bulk_g2s(ip, args.conv + sh * (C::W - 1) * CC, C::CONV_BYTES, bi);
            const uint8_t *gS = reinterpret_cast<const uint8_t *>(args.S) + sh * C::S_BYTES;
            for (int s = 0; s < NST; ++s) {
                mbar_arrive_expect_tx(&bar_S[s], C::ST_BYTES);
                bulk_g2s(smem + s * C::ST_BYTES, gS + (size_t)s * C::ST_BYTES, C::ST_BYTES, &bar_S[s]);
            }
        } else {
            for (int s = 0; s < NST; ++s) mbar_arrive_expect_tx(&bar_S[s], 0);
        }
    };

    if (tid == 0) issue(0, blockIdx.x);

    // Thread 0, on the exit after a timed-out wait in an item: that item's copies (the next item's are issued
    // only after its state has been read) may still be landing in this CTA's shared memory; wait for them,
    // briefly and bounded, before the CTA exits.
    auto drain = [&](int ib, uint32_t par_in, uint32_t par_S) {
        constexpr uint64_t kDrainNs = 10000000ull;
        mbar_wait(&bar_in[ib], par_in, kDrainNs);
        for (int s = 0; s < NST; ++s) mbar_wait(&bar_S[s], par_S, kDrainNs);
    };

    const int g = tid / LPR, cg = tid - (tid / LPR) * LPR;
    for (int it = 0;; ++it) {
        const int item = blockIdx.x + it * gridDim.x;
        if (item >= nitems) break;
        const int ib = it & 1;
        const uint32_t par_in = (uint32_t)(it >> 1) & 1u, par_S = (uint32_t)it & 1u;
        const int n = item / H, h = item - (item / H) * H;
        const int src = __ldg(args.src + n);
        const uint8_t *ip = smem + C::OFF_IN + (size_t)ib * C::IN_BYTES;
        const uint16_t *cs = reinterpret_cast<const uint16_t *>(ip);

        float4 wc[C::CPT];
#pragma unroll
        for (int u = 0; u < C::CPT; ++u) {
            const int c = tid + u * NT;
            if (c < CC) wc[u] = __ldg(reinterpret_cast<const float4 *>(args.conv_w + ((size_t)h * CC + c) * 4));
        }
        const bool fail = !mbar_wait(&bar_in[ib], par_in);
        if (__syncthreads_or(fail)) {
            if (tid == 0) {
                set_status(args.status, KDA_DEV_TIMEOUT);
                drain(ib, par_in, par_S);
            }
            return;
        }
        if (!request_ok(n)) {
            for (int j = 0; j < L; ++j)
                for (int c = tid; c < DV; c += NT) args.y[(((size_t)n * L + j) * H + h) * DV + c] = 0;
            if (tid == 0) set_status(args.status, KDA_DEV_BAD_SLOT);
            __syncthreads();  // every read of the buffers is done
            if (tid == 0) {
                fence_proxy_async_smem();
                issue(ib ^ 1, item + gridDim.x);
            }
            continue;
        }
        // the conv window of this thread's channels, oldest first
        uint16_t w0[C::CPT], w1[C::CPT], w2[C::CPT];
#pragma unroll
        for (int u = 0; u < C::CPT; ++u) {
            const int c = tid + u * NT;
            w0[u] = w1[u] = w2[u] = 0;
            if (c < CC && src >= 0) {
                w0[u] = cs[c];
                w1[u] = cs[CC + c];
                w2[u] = cs[2 * CC + c];
            }
        }
        float4 sr[RPT];  // the state slice, fp32, for all L tokens
        for (int j = 0; j < L; ++j) {
            const size_t th = ((size_t)n * L + j) * H + h;
            const int dj = __ldg(args.dst + (size_t)n * L + j);
            const uint8_t *tp = ip + C::CONV_BYTES + (size_t)j * C::TOK_BYTES;
            const uint16_t *x_s = reinterpret_cast<const uint16_t *>(tp);
            const uint16_t *a_s = reinterpret_cast<const uint16_t *>(tp + C::T_A);
            const uint16_t *z_s = reinterpret_cast<const uint16_t *>(tp + C::T_Z);
            const float beta = sigmoidf_(bf2f(__ldg(args.b + th)));
            // ---- causal conv (+ SiLU); the window after this token goes to the kept slot ----
            uint16_t *cd = dj >= 0 ? args.conv + ((size_t)dj * H + h) * (C::W - 1) * CC : nullptr;
#pragma unroll
            for (int u = 0; u < C::CPT; ++u) {
                const int c = tid + u * NT;
                if (c >= CC) break;
                const uint16_t xr = x_s[c];
                const float4 w = wc[u];
                float acc = w.w * bf2f(xr);
                acc = fmaf(w.x, bf2f(w0[u]), acc);
                acc = fmaf(w.y, bf2f(w1[u]), acc);
                acc = fmaf(w.z, bf2f(w2[u]), acc);
                if (args.silu) acc = acc / (1.0f + __expf(-acc));
                xs[c] = acc;
                w0[u] = w1[u];
                w1[u] = w2[u];
                w2[u] = xr;
                if (cd) {
                    cd[c] = w0[u];
                    cd[CC + c] = w1[u];
                    cd[2 * CC + c] = w2[u];
                }
            }
            float zg = 1.f;
            if (args.z && tid < DV) zg = sigmoidf_(bf2f(z_s[tid]));
            __syncthreads();
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
            // ---- pass 1 over the state: column sums of k^T S' and q^T S' ----
            float4 accK = make_float4(0.f, 0.f, 0.f, 0.f), accQ = accK;
            bool sfail = false;
            if (j == 0) {
                if (src >= 0) {
#pragma unroll
                    for (int s = 0; s < NST; ++s) {
                        sfail |= !mbar_wait(&bar_S[s], par_S);
#pragma unroll
                        for (int m = 0; m < C::M_ST; ++m) {
                            const int mm = s * C::M_ST + m;
                            const int row = g + mm * RPP;
                            if (SBF) {
                                const uint2 hb = *reinterpret_cast<const uint2 *>(smem + (row * DV + cg * 4) * 2);
                                sr[mm] = make_float4(bf2f((uint16_t)(hb.x & 0xffff)), bf2f((uint16_t)(hb.x >> 16)),
                                                     bf2f((uint16_t)(hb.y & 0xffff)), bf2f((uint16_t)(hb.y >> 16)));
                            } else {
                                sr[mm] = *reinterpret_cast<const float4 *>(smem + (row * DV + cg * 4) * 4);
                            }
                        }
                    }
                } else {
#pragma unroll
                    for (int mm = 0; mm < RPT; ++mm) sr[mm] = make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
#pragma unroll
            for (int mm = 0; mm < RPT; ++mm) {
                const int row = g + mm * RPP;
                const float4 x = sr[mm];
                const float kk = ka[row], qq = qa[row];
                accK.x = fmaf(kk, x.x, accK.x); accK.y = fmaf(kk, x.y, accK.y);
                accK.z = fmaf(kk, x.z, accK.z); accK.w = fmaf(kk, x.w, accK.w);
                accQ.x = fmaf(qq, x.x, accQ.x); accQ.y = fmaf(qq, x.y, accQ.y);
                accQ.z = fmaf(qq, x.z, accQ.z); accQ.w = fmaf(qq, x.w, accQ.w);
            }
            *reinterpret_cast<float4 *>(red_k + g * DV + cg * 4) = accK;
            *reinterpret_cast<float4 *>(red_q + g * DV + cg * 4) = accQ;
            if (__syncthreads_or(sfail)) {
                if (tid == 0) {
                    set_status(args.status, KDA_DEV_TIMEOUT);
                    drain(ib, par_in, par_S);
                }
                return;
            }
            if (j == 0 && tid == 0) {  // the state buffer and the other input buffer are free: next item
                fence_proxy_async_smem();
                issue(ib ^ 1, item + gridDim.x);
            }
            for (int c = tid; c < DV; c += NT) {
                float kS = 0.f, qS = 0.f;
#pragma unroll
                for (int r = 0; r < RPP; ++r) {
                    kS += red_k[r * DV + c];
                    qS += red_q[r * DV + c];
                }
                const float u = xs[2 * DK + c] - kS;
                os[c] = args.scale * fmaf(beta * kq, u, qS);
                bu[c] = beta * u;
            }
            __syncthreads();
            const float ss = warp_dot_array(os, os, DV);
            const float rr = rsqrtf(ss * (1.0f / DV) + args.rms_eps);
            for (int c = tid; c < DV; c += NT) args.y[th * DV + c] = f2bf(os[c] * rr * nw[c] * zg);
            // ---- S <- Diag(alpha) S + k^ (beta u)^T in registers; stored when this position is kept ----
            const float4 b4 = *reinterpret_cast<const float4 *>(bu + cg * 4);
            uint8_t *Sd = dj >= 0 ? reinterpret_cast<uint8_t *>(args.S) + ((size_t)dj * H + h) * C::S_BYTES
                                  : nullptr;
#pragma unroll
            for (int mm = 0; mm < RPT; ++mm) {
                const int row = g + mm * RPP;
                const float aa = al[row], kk = kh[row];
                const float4 x = sr[mm];
                float4 o4;
                o4.x = fmaf(kk, b4.x, aa * x.x);
                o4.y = fmaf(kk, b4.y, aa * x.y);
                o4.z = fmaf(kk, b4.z, aa * x.z);
                o4.w = fmaf(kk, b4.w, aa * x.w);
                sr[mm] = o4;
                if (Sd) {
                    if (SBF) {
                        *reinterpret_cast<uint2 *>(Sd + (row * DV + cg * 4) * 2) =
                            make_uint2((uint32_t)f2bf(o4.x) | ((uint32_t)f2bf(o4.y) << 16),
                                       (uint32_t)f2bf(o4.z) | ((uint32_t)f2bf(o4.w) << 16));
                    } else {
                        *reinterpret_cast<float4 *>(Sd + (row * DV + cg * 4) * 4) = o4;
                    }
                }
            }
            __syncthreads();  // xs, kh, al, bu, os and the reductions are rewritten by the next token
        }
    }
}

template <int DK, int DV, bool SBF>
static int launch_multi_t(const DecodeArgs &a, int L, cudaStream_t st) {
    using C = MultiShape<DK, DV, SBF>;
    auto kern = kda_decode_multi_kernel<DK, DV, SBF>;
    static int occ_cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return launch_result("decode_multi: cudaGetDevice");
    if (occ_cache[dev] == 0) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
            return launch_result("decode_multi: cudaFuncSetAttribute");
        int occ = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, C::NT, C::SMEM) != cudaSuccess || occ < 1)
            return fail(KDA_ERR_CUDA, "decode_multi: the kernel cannot be resident on this device");
        occ_cache[dev] = occ;
    }
    const int items = a.n * a.H;
    const int cap = current_device_sms() * occ_cache[dev];
    const int grid = items < cap ? items : cap;
    kern<<<grid, C::NT, C::SMEM, st>>>(a, L);
    return launch_result("kda_decode_multi_kernel launch");
}

template <int DK, int DV>
static int launch_multi_dt(const DecodeArgs &a, int L, cudaStream_t st) {
    return a.state_bf16 ? launch_multi_t<DK, DV, true>(a, L, st) : launch_multi_t<DK, DV, false>(a, L, st);
}

int launch_decode_multi(const DecodeArgs &a, int dk, int dv, int L, cudaStream_t st) {
    if (dk == 128 && dv == 128) return launch_multi_dt<128, 128>(a, L, st);
    if (dk == 64 && dv == 64) return launch_multi_dt<64, 64>(a, L, st);
    if (dk == 32 && dv == 16) return launch_multi_dt<32, 16>(a, L, st);
    if (dk == 16 && dv == 32) return launch_multi_dt<16, 32>(a, L, st);
    if (dk == 16 && dv == 16) return launch_multi_dt<16, 16>(a, L, st);
    return fail(KDA_ERR_UNSUPPORTED_SHAPE, "decode_multi: (dk, dv) not compiled in");
}

}  // namespace kda
