// kda_prefill.cu -- chunked KDA prefill with checkpoint emission into the state-slot pool.
//
// Chunked WY/UT form of the gated delta rule with channel-wise decay ("A Preview of Production-Scale
// Kimi K3 Support on vLLM", section "KDA prefill and decode": chunked prefill with the initial states
// gathered in one operation; section "The Hardest Part: Prefix Caching for KDA": the state must exist at
// the exact prefix boundary).  For a chunk of n tokens starting from state S0, with G_r the cumulative
// log-decay inside the chunk (row r included):
//     A_rs  = sum_i k_ri k_si exp(G_ri - G_si)            (s < r)
//     Qk_rs = scale * sum_i q_ri k_si exp(G_ri - G_si)    (s <= r)
//     [W | U'] = (I + diag(beta) A)^{-1} diag(beta) [k * exp(G) | v]
//     U = U' - W S0,   O = scale * (q * exp(G)) S0 + Qk U,   S1 = Diag(exp(G_last)) S0 + (k * exp(G_last - G))^T U
// Chunks are aligned to absolute token positions (start_pos + i), so a sequence resumed at a chunk
// boundary performs exactly the arithmetic of a full replay from that boundary on.
//
// Launches (one stream, graph-capturable):
//   1. table:  validates cu_seqlens / start_pos / checkpoint offsets, builds the chunk table;
//   2. intra:  one CTA per (chunk, head): causal conv + SiLU, L2 norms, gates, A, Qk, the unit-lower
//              triangular solve, W / U' / decayed K / decayed Q into the workspace; conv windows of
//              checkpoints and of the final state go straight to the pool;
//   3. state:  one CTA per (sequence, head, dv tile), sequential over the sequence's chunks: U, O and the
//              state chain in fp32; checkpoint states written at every boundary, the final one to dst;
//   4. out:    gated RMSNorm of O into the bf16 output.
#include <algorithm>

#include "kda_device.cuh"
#include "kda_internal.h"
#include "kda_umma.cuh"

namespace kda {

namespace {

constexpr int kConvW = 4;
constexpr int kThreads = 256;
constexpr int kMaxSeqThreads = 1024;

struct ChunkEnt {
    int32_t seq, t0, n, ord;  // sequence, first token index, tokens, chunk ordinal within the sequence
};

enum : int32_t { kSeqInvalid = 1, kSeqCkptBad = 2 };

struct Layout {
    int64_t maxc;
    size_t off_cnt, off_ent, off_pos, off_seqc, off_flags;
    size_t off_W, off_U, off_Kt, off_Qp, off_Qk, off_gl, off_O;
    size_t total;
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

Layout make_layout(int H, int dk, int dv, int nseq, int64_t T, int C) {
    Layout L;
    L.maxc = T / C + 2 * (int64_t)nseq + 1;
    size_t o = 0;
    L.off_cnt = o; o = align256(o + 16);
    L.off_ent = o; o = align256(o + sizeof(ChunkEnt) * L.maxc);
    L.off_pos = o; o = align256(o + sizeof(int64_t) * L.maxc);
    L.off_seqc = o; o = align256(o + sizeof(int32_t) * (nseq + 1));
    L.off_flags = o; o = align256(o + sizeof(int32_t) * (nseq + 1));
    const size_t per = (size_t)L.maxc * H;
    L.off_W = o; o = align256(o + 4 * per * C * dk);
    L.off_U = o; o = align256(o + 4 * per * C * dv);
    L.off_Kt = o; o = align256(o + 4 * per * C * dk);
    L.off_Qp = o; o = align256(o + 4 * per * C * dk);
    L.off_Qk = o; o = align256(o + 4 * per * C * C);
    L.off_gl = o; o = align256(o + 4 * per * dk);
    L.off_O = o; o = align256(o + 4 * (size_t)T * H * dv);
    L.total = o;
    return L;
}

template <typename T>
__device__ __forceinline__ T *wsp(const PrefillArgs &a, size_t off) {
    return reinterpret_cast<T *>(reinterpret_cast<uint8_t *>(a.ws) + off);
}

__device__ __forceinline__ float log_sigmoid(float x) {
    return x < 0.f ? x - log1pf(expf(x)) : -log1pf(expf(-x));
}

// Raw q|k|v input of channel ch for token t of head h (bf16 -> fp32).
__device__ __forceinline__ float raw_input(const PrefillArgs &a, int dk, int dv, int64_t t, int h, int ch) {
    const int H = a.H;
    if (ch < dk) return bf2f(a.q[((size_t)t * H + h) * dk + ch]);
    if (ch < 2 * dk) return bf2f(a.k[((size_t)t * H + h) * dk + (ch - dk)]);
    return bf2f(a.v[((size_t)t * H + h) * dv + (ch - 2 * dk)]);
}

__device__ __forceinline__ uint16_t raw_bits(const PrefillArgs &a, int dk, int dv, int64_t t, int h, int ch) {
    const int H = a.H;
    if (ch < dk) return a.q[((size_t)t * H + h) * dk + ch];
    if (ch < 2 * dk) return a.k[((size_t)t * H + h) * dk + (ch - dk)];
    return a.v[((size_t)t * H + h) * dv + (ch - 2 * dk)];
}

// Raw bits of channel ch at absolute position pos of sequence n (pos >= start - (W-1)): from this
// call's tokens when pos >= start, else from the source slot's stored window (zeros for src = -1).
__device__ __forceinline__ uint16_t raw_at(const PrefillArgs &a, int dk, int dv, int h, int ch, int64_t pos,
                                           int64_t start, int64_t ts, int src) {
    if (pos >= start) return raw_bits(a, dk, dv, ts + (pos - start), h, ch);
    if (src < 0) return 0;
    const int CC = 2 * dk + dv;
    const int row = (int)(pos - start + (kConvW - 1));
    return a.conv[(((size_t)src * a.H + h) * (kConvW - 1) + row) * CC + ch];
}

// ------------------------------------------------------------------------------------------ 1. table
__global__ void __launch_bounds__(kMaxSeqThreads) prefill_table_kernel(const PrefillArgs a, const Layout L) {
    __shared__ int32_t scan[kMaxSeqThreads];
    __shared__ int32_t carry_s;
    const int tid = threadIdx.x;
    const int C = a.chunk;
    int32_t *cnt = wsp<int32_t>(a, L.off_cnt);
    int32_t *seqc = wsp<int32_t>(a, L.off_seqc);
    int32_t *flags = wsp<int32_t>(a, L.off_flags);
    if (tid == 0) carry_s = 0;
    __syncthreads();
    for (int base = 0; base < a.nseq; base += kMaxSeqThreads) {
        const int n = base + tid;
        int32_t c = 0;
        if (n < a.nseq) {
            const int64_t t0 = a.cu_seqlens[n], t1 = a.cu_seqlens[n + 1];
            const int64_t start = a.start_pos[n];
            bool ok = t0 >= 0 && t1 >= t0 && t1 <= a.total_tokens && start >= 0;
            if (n == 0 && t0 != 0) ok = false;
            if (n == a.nseq - 1 && t1 != a.total_tokens) ok = false;
            const int src = a.src[n], dst = a.dst[n];
            const bool slots_ok = src >= -1 && src < a.num_slots && dst >= 0 && dst < a.num_slots;
            int32_t f = 0;
            if (!ok || !slots_ok) {
                f = kSeqInvalid;
                set_status(a.status, ok ? KDA_DEV_BAD_SLOT : KDA_DEV_BAD_SEQLENS);
            } else {
                const int64_t len = t1 - t0;
                c = len > 0 ? (int32_t)((start + len + C - 1) / C - start / C) : 0;
                if (a.interval > 0) {
                    const int64_t expect = (start + len) / a.interval - start / a.interval;
                    if ((int64_t)a.ckpt_offsets[n + 1] - a.ckpt_offsets[n] != expect || a.ckpt_offsets[n] < 0) {
                        f |= kSeqCkptBad;
                        set_status(a.status, KDA_DEV_BAD_CKPT);
                    }
                }
            }
            flags[n] = f;
        }
        scan[tid] = c;
        __syncthreads();
        for (int o = 1; o < kMaxSeqThreads; o <<= 1) {  // inclusive Hillis-Steele scan
            const int32_t v = tid >= o ? scan[tid - o] : 0;
            __syncthreads();
            scan[tid] += v;
            __syncthreads();
        }
        if (n < a.nseq) seqc[n] = carry_s + scan[tid] - c;
        __syncthreads();
        if (tid == kMaxSeqThreads - 1) carry_s += scan[tid];
        __syncthreads();
    }
    if (tid == 0) {
        seqc[a.nseq] = carry_s;
        cnt[0] = carry_s;
    }
    __syncthreads();
    const int32_t total = carry_s;
    ChunkEnt *ent = wsp<ChunkEnt>(a, L.off_ent);
    int64_t *pos = wsp<int64_t>(a, L.off_pos);
    for (int32_t c = tid; c < total; c += kMaxSeqThreads) {
        int lo = 0, hi = a.nseq - 1;  // last sequence with seqc[n] <= c
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (seqc[mid] <= c) lo = mid; else hi = mid - 1;
        }
        const int n = lo;
        const int32_t j = c - seqc[n];
        const int64_t start = a.start_pos[n];
        const int64_t len = (int64_t)a.cu_seqlens[n + 1] - a.cu_seqlens[n];
        const int64_t p0 = j == 0 ? start : (start / C + j) * C;
        int64_t p1 = (start / C + j + 1) * C;
        if (p1 > start + len) p1 = start + len;
        ChunkEnt e;
        e.seq = n;
        e.t0 = (int32_t)(a.cu_seqlens[n] + (p0 - start));
        e.n = (int32_t)(p1 - p0);
        e.ord = j;
        ent[c] = e;
        pos[c] = p0;
    }
}

// ------------------------------------------------------------------------------------------ 2. intra
__global__ void __launch_bounds__(kThreads) prefill_intra_kernel(const PrefillArgs a, const Layout L, int dk, int dv) {
    extern __shared__ __align__(16) float sm[];
    const int C = a.chunk, H = a.H, CC = 2 * dk + dv, DY = dk + dv;
    const int c = blockIdx.x, h = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (c >= *wsp<int32_t>(a, L.off_cnt)) return;
    const ChunkEnt e = wsp<ChunkEnt>(a, L.off_ent)[c];
    const int64_t p0 = wsp<int64_t>(a, L.off_pos)[c];
    const int n = e.seq, ntok = e.n;
    const int64_t start = a.start_pos[n], ts = a.cu_seqlens[n];
    const int64_t len = (int64_t)a.cu_seqlens[n + 1] - ts;
    const int srcv = a.src[n];  // validated by the table kernel (sequences with bad slots have no chunks)

    float *qh = sm;                // [C][dk]
    float *kh = qh + C * dk;       // [C][dk]
    float *G = kh + C * dk;        // [C][dk]
    float *Y = G + C * dk;         // [C][dk + dv]  (k*exp(G) | v), solved in place into (W | U')
    float *A = Y + C * DY;         // [C][C]
    float *Qk = A + C * C;         // [C][C]
    float *beta = Qk + C * C;      // [C]

    // causal conv + SiLU, one channel per thread, sequential over the chunk's tokens
    for (int ch = tid; ch < CC; ch += kThreads) {
        float hist[kConvW - 1];
        for (int j = 0; j < kConvW - 1; ++j) hist[j] = bf2f(raw_at(a, dk, dv, h, ch, p0 - (kConvW - 1) + j, start, ts, srcv));
        const float4 w = __ldg(reinterpret_cast<const float4 *>(a.conv_w + ((size_t)h * CC + ch) * kConvW));
        for (int r = 0; r < C; ++r) {
            float out = 0.f;
            if (r < ntok) {
                const float x = raw_input(a, dk, dv, e.t0 + r, h, ch);
                out = w.w * x;
                out = fmaf(w.x, hist[0], out);
                out = fmaf(w.y, hist[1], out);
                out = fmaf(w.z, hist[2], out);
                if (a.silu) out = out / (1.f + __expf(-out));
                hist[0] = hist[1];
                hist[1] = hist[2];
                hist[2] = x;
            }
            if (ch < dk) qh[r * dk + ch] = out;
            else if (ch < 2 * dk) kh[r * dk + ch - dk] = out;
            else Y[r * DY + dk + (ch - 2 * dk)] = out;
        }
    }
    // gates: log alpha (0 for padding rows) and beta (0 for padding rows)
    for (int idx = tid; idx < C * dk; idx += kThreads) {
        const int r = idx / dk, i = idx - (idx / dk) * dk;
        G[idx] = r < ntok ? log_sigmoid(bf2f(a.a[((size_t)(e.t0 + r) * H + h) * dk + i])) : 0.f;
    }
    for (int r = tid; r < C; r += kThreads) beta[r] = r < ntok ? sigmoidf_(bf2f(a.b[(size_t)(e.t0 + r) * H + h])) : 0.f;
    __syncthreads();
    // L2 norms of q and k per token (one warp per token)
    for (int r = warp; r < ntok; r += kThreads / 32) {
        const float nq = warp_dot_array(qh + r * dk, qh + r * dk, dk);
        const float nk = warp_dot_array(kh + r * dk, kh + r * dk, dk);
        const float rq = rsqrtf(nq + a.l2_eps), rk = rsqrtf(nk + a.l2_eps);
        for (int i = lane; i < dk; i += 32) {
            qh[r * dk + i] *= rq;
            kh[r * dk + i] *= rk;
        }
    }
    // cumulative log decay along the chunk
    for (int i = tid; i < dk; i += kThreads) {
        float acc = 0.f;
        for (int r = 0; r < C; ++r) {
            acc += G[r * dk + i];
            G[r * dk + i] = acc;
        }
    }
    __syncthreads();
    for (int idx = tid; idx < C * dk; idx += kThreads) {
        const int r = idx / dk, i = idx - (idx / dk) * dk;
        Y[r * DY + i] = kh[idx] * expf(G[idx]);
    }
    // A (strict lower) and scaled Qk (lower with diagonal), exact pairwise exponentials
    for (int idx = tid; idx < C * C; idx += kThreads) {
        const int r = idx / C, s = idx - (idx / C) * C;
        float accA = 0.f, accQ = 0.f;
        if (s <= r && r < ntok) {
            for (int i = 0; i < dk; ++i) {
                const float d = __expf(G[r * dk + i] - G[s * dk + i]);
                const float ks = kh[s * dk + i] * d;
                accA = fmaf(kh[r * dk + i], ks, accA);
                accQ = fmaf(qh[r * dk + i], ks, accQ);
            }
        }
        A[idx] = s < r ? accA : 0.f;
        Qk[idx] = a.scale * accQ;
    }
    __syncthreads();
    // forward substitution, one column per thread: x_r = beta_r (y_r - sum_{s<r} A_rs x_s)
    for (int col = tid; col < DY; col += kThreads) {
        for (int r = 0; r < C; ++r) {
            float acc = Y[r * DY + col];
            for (int s = 0; s < r; ++s) acc = fmaf(-A[r * C + s], Y[s * DY + col], acc);
            Y[r * DY + col] = beta[r] * acc;
        }
    }
    __syncthreads();
    const size_t cb = (size_t)c * H + h;
    float *gW = wsp<float>(a, L.off_W) + cb * C * dk;
    float *gU = wsp<float>(a, L.off_U) + cb * C * dv;
    float *gKt = wsp<float>(a, L.off_Kt) + cb * C * dk;
    float *gQp = wsp<float>(a, L.off_Qp) + cb * C * dk;
    float *gQk = wsp<float>(a, L.off_Qk) + cb * C * C;
    float *ggl = wsp<float>(a, L.off_gl) + cb * dk;
    const float *Glast = G + (C - 1) * dk;
    for (int idx = tid; idx < C * dk; idx += kThreads) {
        const int r = idx / dk, i = idx - (idx / dk) * dk;
        gW[idx] = Y[r * DY + i];
        gKt[idx] = kh[idx] * expf(Glast[i] - G[idx]);
        gQp[idx] = a.scale * qh[idx] * expf(G[idx]);
    }
    for (int idx = tid; idx < C * dv; idx += kThreads) {
        const int r = idx / dv, j = idx - (idx / dv) * dv;
        gU[idx] = Y[r * DY + dk + j];
    }
    for (int idx = tid; idx < C * C; idx += kThreads) gQk[idx] = Qk[idx];
    for (int i = tid; i < dk; i += kThreads) ggl[i] = expf(Glast[i]);

    // raw conv windows at a checkpoint boundary / at the sequence end go straight to the pool
    const int32_t flag = wsp<int32_t>(a, L.off_flags)[n];
    const int64_t pend = p0 + ntok;
    int wslot[2] = {-1, -1};
    if (a.interval > 0 && pend % a.interval == 0 && !(flag & kSeqCkptBad)) {
        const int64_t j = pend / a.interval - start / a.interval - 1;
        const int s = a.ckpt_slots[a.ckpt_offsets[n] + j];
        if (s >= a.num_slots || s < -1) {
            if (tid == 0) set_status(a.status, KDA_DEV_BAD_SLOT);
        } else {
            wslot[0] = s;
        }
    }
    if (pend == start + len) wslot[1] = a.dst[n];
    for (int w = 0; w < 2; ++w) {
        if (wslot[w] < 0) continue;
        uint16_t *cw = a.conv + ((size_t)wslot[w] * H + h) * (kConvW - 1) * CC;
        for (int idx = tid; idx < (kConvW - 1) * CC; idx += kThreads) {
            const int row = idx / CC, ch = idx - (idx / CC) * CC;
            cw[idx] = raw_at(a, dk, dv, h, ch, pend - (kConvW - 1) + row, start, ts, srcv);
        }
    }
}

// ------------------------------------------------------------------------------------------ 3. state
__global__ void __launch_bounds__(kThreads) prefill_state_kernel(const PrefillArgs a, const Layout L, int dk, int dv,
                                                                  int DVT) {
    extern __shared__ __align__(16) float sm[];
    const int C = a.chunk, H = a.H;
    const int n = blockIdx.x, h = blockIdx.y, j0 = blockIdx.z * DVT, tid = threadIdx.x;
    const int32_t flag = wsp<int32_t>(a, L.off_flags)[n];
    if (flag & kSeqInvalid) return;
    const int src = a.src[n], dst = a.dst[n];  // validated by the table kernel
    float *S = sm;                 // [dk][DVT]
    float *Wm = S + dk * DVT;      // [C][dk]
    float *Kt = Wm + C * dk;       // [C][dk]
    float *Qp = Kt + C * dk;       // [C][dk]
    float *Qk = Qp + C * dk;       // [C][C]
    float *Ut = Qk + C * C;        // [C][DVT]
    float *U = Ut + C * DVT;       // [C][DVT]
    float *gl = U + C * DVT;       // [dk]
    for (int idx = tid; idx < dk * DVT; idx += kThreads) {
        const int i = idx / DVT, j = idx - (idx / DVT) * DVT;
        S[idx] = src >= 0 ? load_state(a.S, a.state_bf16, (((size_t)src * H + h) * dk + i) * dv + j0 + j) : 0.f;
    }
    const int64_t start = a.start_pos[n];
    const int32_t c0 = wsp<int32_t>(a, L.off_seqc)[n], c1 = wsp<int32_t>(a, L.off_seqc)[n + 1];
    const ChunkEnt *ent = wsp<ChunkEnt>(a, L.off_ent);
    const int64_t *pos = wsp<int64_t>(a, L.off_pos);
    float *gO = wsp<float>(a, L.off_O);
    __syncthreads();
    for (int32_t c = c0; c < c1; ++c) {
        const ChunkEnt e = ent[c];
        const size_t cb = (size_t)c * H + h;
        const float *gW = wsp<float>(a, L.off_W) + cb * C * dk;
        const float *gU = wsp<float>(a, L.off_U) + cb * C * dv;
        const float *gKt = wsp<float>(a, L.off_Kt) + cb * C * dk;
        const float *gQp = wsp<float>(a, L.off_Qp) + cb * C * dk;
        const float *gQk = wsp<float>(a, L.off_Qk) + cb * C * C;
        const float *ggl = wsp<float>(a, L.off_gl) + cb * dk;
        for (int idx = tid; idx < C * dk; idx += kThreads) {
            Wm[idx] = gW[idx];
            Kt[idx] = gKt[idx];
            Qp[idx] = gQp[idx];
        }
        for (int idx = tid; idx < C * C; idx += kThreads) Qk[idx] = gQk[idx];
        for (int idx = tid; idx < C * DVT; idx += kThreads) {
            const int r = idx / DVT, j = idx - (idx / DVT) * DVT;
            Ut[idx] = gU[r * dv + j0 + j];
        }
        for (int i = tid; i < dk; i += kThreads) gl[i] = ggl[i];
        __syncthreads();
        // U = U' - W S
        for (int idx = tid; idx < C * DVT; idx += kThreads) {
            const int r = idx / DVT, j = idx - (idx / DVT) * DVT;
            float acc = Ut[idx];
            for (int i = 0; i < dk; ++i) acc = fmaf(-Wm[r * dk + i], S[i * DVT + j], acc);
            U[idx] = acc;
        }
        __syncthreads();
        // O = Q+ S + Qk U  (scale folded into Q+ and Qk)
        for (int idx = tid; idx < C * DVT; idx += kThreads) {
            const int r = idx / DVT, j = idx - (idx / DVT) * DVT;
            if (r >= e.n) continue;
            float acc = 0.f;
            for (int i = 0; i < dk; ++i) acc = fmaf(Qp[r * dk + i], S[i * DVT + j], acc);
            for (int s = 0; s <= r; ++s) acc = fmaf(Qk[r * C + s], U[s * DVT + j], acc);
            gO[((size_t)(e.t0 + r) * H + h) * dv + j0 + j] = acc;
        }
        __syncthreads();
        // S = Diag(exp(G_last)) S + Kt^T U
        for (int idx = tid; idx < dk * DVT; idx += kThreads) {
            const int i = idx / DVT, j = idx - (idx / DVT) * DVT;
            float acc = gl[i] * S[idx];
            for (int r = 0; r < C; ++r) acc = fmaf(Kt[r * dk + i], U[r * DVT + j], acc);
            S[idx] = acc;
        }
        __syncthreads();
        const int64_t pend = pos[c] + e.n;
        if (a.interval > 0 && pend % a.interval == 0 && !(flag & kSeqCkptBad)) {
            const int64_t j = pend / a.interval - start / a.interval - 1;
            const int s = a.ckpt_slots[a.ckpt_offsets[n] + j];
            if (s >= 0 && s < a.num_slots) {
                for (int idx = tid; idx < dk * DVT; idx += kThreads) {
                    const int i = idx / DVT, jj = idx - (idx / DVT) * DVT;
                    store_state(a.S, a.state_bf16, (((size_t)s * H + h) * dk + i) * dv + j0 + jj, S[idx]);
                }
            }
        }
    }
    for (int idx = tid; idx < dk * DVT; idx += kThreads) {
        const int i = idx / DVT, j = idx - (idx / DVT) * DVT;
        store_state(a.S, a.state_bf16, (((size_t)dst * H + h) * dk + i) * dv + j0 + j, S[idx]);
    }
    if (c0 == c1 && blockIdx.z == 0) {  // empty sequence: the window passes through unchanged
        const int CC = 2 * dk + dv;
        uint16_t *cw = a.conv + ((size_t)dst * H + h) * (kConvW - 1) * CC;
        for (int idx = tid; idx < (kConvW - 1) * CC; idx += kThreads)
            cw[idx] = src >= 0 ? a.conv[((size_t)src * H + h) * (kConvW - 1) * CC + idx] : (uint16_t)0;
    }
}

// ------------------------------------------------------------------------------------------ 4. output
__global__ void __launch_bounds__(kThreads) prefill_out_kernel(const PrefillArgs a, const Layout L, int dv) {
    const int H = a.H, C = a.chunk;
    const int c = blockIdx.x, h = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (c >= *wsp<int32_t>(a, L.off_cnt)) return;
    const ChunkEnt e = wsp<ChunkEnt>(a, L.off_ent)[c];
    const float *gO = wsp<float>(a, L.off_O);
    for (int r = warp; r < e.n && r < C; r += kThreads / 32) {
        const size_t base = ((size_t)(e.t0 + r) * H + h) * dv;
        float ss = 0.f;
        for (int j = lane; j < dv; j += 32) ss = fmaf(gO[base + j], gO[base + j], ss);
        ss = warp_sum(ss);
        const float rr = rsqrtf(ss / dv + a.rms_eps);
        for (int j = lane; j < dv; j += 32) {
            float yv = gO[base + j] * rr * __ldg(a.norm_w + j);
            if (a.z) yv *= sigmoidf_(bf2f(a.z[base + j]));
            a.y[base + j] = f2bf(yv);
        }
    }
}

// ================================================================================ tensor-core path
// dk = dv = 128, chunk 64.  Transposed formulation so that every MMA has M = 128 (TMEM lane = row):
//   [A ; Qk]  = [K+ ; Q+] (mid-chunk reference) x K-^T           bf16, M=128 N=64  K=128
//   W^T       = (k*exp(G))^T x T^T,   U'^T = V^T x T^T            tf32, M=128 N=64  K=64
//   U^T       = U'^T + S^T x (-W)^T                                bf16, M=128 N=64  K=128
//   O^T       = S^T x Q+^T + U^T x Qk^T                            bf16, M=128 N=64  K=128 / 64
//   S^T       = S^T Diag(exp(G_last)) + U^T x Ktil                 tf32, M=128 N=128 K=64
// tf32 operands are rounded to nearest (cvt.rna); accumulation is fp32 in tensor memory.
namespace tc {

constexpr int D = 128, CH = 64, NT = 256;
constexpr float kMidRange = 40.f;  // |G_r - G_mid| bound for the factorised A / Qk (fp32-safe)

// Workspace block per (chunk, head); the first WS_OPS bytes are operand tiles in their shared-memory
// layout (K-major, 128B swizzle), copied verbatim by the state kernel.
constexpr uint32_t WS_QK = 0;                    // bf16 [64 r][64 s]    Qk (scaled, masked)
constexpr uint32_t WS_W = WS_QK + CH * CH * 2;   // bf16 [64 r][128 i]   -W (negated)
constexpr uint32_t WS_QP = WS_W + CH * D * 2;    // bf16 [64 r][128 i]   scale * q * exp(G)
constexpr uint32_t WS_KT = WS_QP + CH * D * 2;   // tf32 [128 i][64 r]   k * exp(G_last - G), transposed
constexpr uint32_t WS_GL = WS_KT + D * CH * 4;   // fp32 [128]           exp(G_last)
constexpr uint32_t WS_OPS = WS_GL + D * 4;
constexpr uint32_t WS_UP = (WS_OPS + 255) / 256 * 256;  // fp32 [64 r][128 j]   U'
constexpr uint32_t WS_BLOCK = WS_UP + CH * D * 4;
static_assert(WS_W % 1024 == 0 && WS_QP % 1024 == 0 && WS_KT % 1024 == 0 && WS_GL % 1024 == 0, "tile align");
static_assert(WS_OPS % 16 == 0, "bulk copy size");

struct Layout2 {
    int64_t maxc;
    size_t off_cnt, off_ent, off_pos, off_seqc, off_flags, off_blk, total;
};

inline Layout2 make_layout2(int H, int nseq, int64_t T) {
    Layout2 L;
    L.maxc = T / CH + 2 * (int64_t)nseq + 1;
    size_t o = 0;
    L.off_cnt = o; o = align256(o + 16);
    L.off_ent = o; o = align256(o + sizeof(ChunkEnt) * L.maxc);
    L.off_pos = o; o = align256(o + sizeof(int64_t) * L.maxc);
    L.off_seqc = o; o = align256(o + sizeof(int32_t) * (nseq + 1));
    L.off_flags = o; o = align256(o + sizeof(int32_t) * (nseq + 1));
    o = (o + 1023) & ~size_t(1023);
    L.off_blk = o; o += (size_t)WS_BLOCK * L.maxc * H;
    L.total = o;
    return L;
}

inline Layout as_layout(const Layout2 &L2) {  // the table kernel only uses these fields
    Layout L{};
    L.maxc = L2.maxc;
    L.off_cnt = L2.off_cnt; L.off_ent = L2.off_ent; L.off_pos = L2.off_pos;
    L.off_seqc = L2.off_seqc; L.off_flags = L2.off_flags;
    return L;
}

__device__ __forceinline__ bool wait_all(uint64_t *bar, uint32_t parity) {
    const bool ok = mbar_wait(bar, parity);
    return __syncthreads_or(!ok) == 0;
}

// Intra-chunk kernel smem (bytes, from a 1024-aligned base), by phase:
//   P0-P1  [0,32K) q^ fp32 | [32K,64K) k^ fp32 | [64K,96K) G fp32 | [96K,128K) V^T tf32 tile | [128K,180K) raw rows
//   P2     [128K,160K) [K+;Q+] bf16 tile | [160K,176K) K- bf16 tile
//   P3-P4  [0,8K) Qk staging, then [0,16K) Inv fp32 | [128K,145K) A fp32 (row stride 68) | [160K,176K) block temps,
//          then T tf32
//   P5     [0,32K) (k exp G)^T tf32 tile | [128K,160K) Ktil^T tf32 staging
//   P6     [32K,48K) -W bf16 staging | [64K,96K) U' fp32 staging
constexpr uint32_t I_Q = 0, I_K = 32768, I_G = 65536, I_VT = 98304, I_RAW = 131072;
constexpr uint32_t I_X1 = 131072, I_KM = 163840, I_A = 131072, I_T = 163840;
constexpr uint32_t I_INV = 0;          // Inv fp32 [64][64] over q^ (free after the Qk copy-out)
constexpr uint32_t I_QKS_SLOW = 148480; // Qk staging of the wide-decay path (q^ is still read there)
constexpr uint32_t I_MISC = 184320;   // beta, exp(G_mid), decay partial sums, barrier, tmem address, window stash
constexpr uint32_t I_SMEM = I_MISC + 6144 + 1024;  // + alignment slack
constexpr int RAW_ROWS = CH + kConvW - 1;           // 3 history rows + 64 tokens
constexpr int AST = 68;                             // row stride of A in smem (padded against bank conflicts)
static_assert(I_A + CH * AST * 4 <= I_QKS_SLOW && I_QKS_SLOW + CH * CH * 2 <= I_T, "A and slow Qk staging");
static_assert(I_RAW + RAW_ROWS * 3 * D * 2 <= I_MISC, "raw staging");

constexpr int NTI = 512;  // intra kernel threads

__device__ __forceinline__ float log_sigmoid_fast(float x) {
    // log(sigmoid(x)) = min(x, 0) - log(1 + exp(-|x|)); absolute error ~1e-7, which is what the
    // cumulative decay (a sum of these) needs
    return fminf(x, 0.f) - __logf(1.f + __expf(-fabsf(x)));
}

__global__ void __launch_bounds__(NTI, 1) prefill_intra_tc_kernel(const PrefillArgs a, const Layout2 L) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int H = a.H, CC = 3 * D;
    const int c = blockIdx.x, h = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (c >= *wsp<int32_t>(a, L.off_cnt)) return;
    const ChunkEnt e = wsp<ChunkEnt>(a, L.off_ent)[c];
    const int64_t p0 = wsp<int64_t>(a, L.off_pos)[c];
    const int n = e.seq, ntok = e.n;
    const int64_t start = a.start_pos[n], ts = a.cu_seqlens[n];
    const int64_t len = (int64_t)a.cu_seqlens[n + 1] - ts;
    const int srcv = a.src[n];

    float *qh = reinterpret_cast<float *>(sm + I_Q);
    float *kh = reinterpret_cast<float *>(sm + I_K);
    float *G = reinterpret_cast<float *>(sm + I_G);
    uint8_t *Vt = sm + I_VT;
    uint16_t *raw = reinterpret_cast<uint16_t *>(sm + I_RAW);  // [67][384] bf16, row = position p0 - 3 + row
    float *beta = reinterpret_cast<float *>(sm + I_MISC);
    float *eGm = beta + 64;     // exp(G_mid) per channel
    float *gtot = eGm + D;      // [4][128] partial sums of the cumulative decay
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + I_MISC + 3072);
    uint32_t *tmem_s = reinterpret_cast<uint32_t *>(sm + I_MISC + 3136);
    uint8_t *blk = reinterpret_cast<uint8_t *>(a.ws) + L.off_blk + ((size_t)c * H + h) * WS_BLOCK;

    if (warp == 0) umma::alloc(tmem_s, 256);
    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }

    // ---- P0: the chunk's raw q|k|v rows (and 3 rows of history) and decay logits into smem ----
    // One 256-byte bulk copy per (row, tensor), issued by one thread each; rows without a source are
    // zero-filled with ordinary stores.  Row `row` holds position p0 - 3 + row; history rows before the
    // sequence start come from the source slot's stored window.
    uint16_t *astage = reinterpret_cast<uint16_t *>(sm + I_VT);  // decay logits bf16 [64][128] (V^T comes later)
    uint64_t *bar_in = bar + 1;
    const int nrows = (kConvW - 1) + ntok;                        // rows with data
    const int hist_src = (int)min((int64_t)nrows, max((int64_t)0, start - p0 + (kConvW - 1)));  // rows before start
    if (tid == 0) {
        mbar_init(bar_in, 1);
        fence_mbar_init();
        const uint32_t bytes = (uint32_t)((nrows - (srcv >= 0 ? 0 : hist_src)) * 3 * 256 + ntok * 256);
        mbar_arrive_expect_tx(bar_in, bytes);
    }
    __syncthreads();
    if (tid < RAW_ROWS * 3) {
        const int row = tid / 3, part = tid - (tid / 3) * 3;
        const int64_t p = p0 - (kConvW - 1) + row;
        uint16_t *dst = raw + row * CC + part * D;
        const uint16_t *src = nullptr;
        if (row < nrows) {
            if (p >= start) {
                const size_t t = (size_t)(ts + (p - start)) * H + h;
                src = (part == 0 ? a.q : (part == 1 ? a.k : a.v)) + t * D;
            } else if (srcv >= 0) {
                src = a.conv + (((size_t)srcv * H + h) * (kConvW - 1) + (p - start + (kConvW - 1))) * CC + part * D;
            }
        }
        if (src) {
            bulk_g2s(dst, src, 256, bar_in);
        } else {
            uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
            for (int u = 0; u < 16; ++u) d4[u] = make_uint4(0u, 0u, 0u, 0u);
        }
    } else if (tid >= 256 && tid < 256 + CH) {
        const int r = tid - 256;
        uint16_t *dst = astage + r * D;
        if (r < ntok) {
            bulk_g2s(dst, a.a + ((size_t)(e.t0 + r) * H + h) * D, 256, bar_in);
        } else {
            uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
            for (int u = 0; u < 16; ++u) d4[u] = make_uint4(0u, 0u, 0u, 0u);
        }
    }
    if (__syncthreads_or(!mbar_wait(bar_in, 0))) {
        if (tid == 0) set_status(a.status, KDA_DEV_TIMEOUT);
        __syncthreads();
        if (warp == 0) umma::dealloc(*tmem_s, 256);
        return;
    }
    for (int idx = tid; idx < CH * 16; idx += NTI) {  // log decay, 8 channels per item
        const int r = idx >> 4, part = idx & 15;
        const uint4 v = reinterpret_cast<const uint4 *>(astage + r * D)[part];
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
        float g8[8];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            g8[2 * q] = r < ntok ? log_sigmoid_fast(bf2f((uint16_t)(w4[q] & 0xffff))) : 0.f;
            g8[2 * q + 1] = r < ntok ? log_sigmoid_fast(bf2f((uint16_t)(w4[q] >> 16))) : 0.f;
        }
        float4 *gd = reinterpret_cast<float4 *>(G + r * D + part * 8);
        gd[0] = make_float4(g8[0], g8[1], g8[2], g8[3]);
        gd[1] = make_float4(g8[4], g8[5], g8[6], g8[7]);
    }
    if (tid < CH) beta[tid] = tid < ntok ? sigmoidf_(bf2f(a.b[(size_t)(e.t0 + tid) * H + h])) : 0.f;
    __syncthreads();
    // ---- P1: causal conv + SiLU, one channel per thread along the chunk (window in registers) ----
    if (tid < CC) {
        const int ch = tid;
        const float4 w = __ldg(reinterpret_cast<const float4 *>(a.conv_w + ((size_t)h * CC + ch) * kConvW));
        float h0 = bf2f(raw[ch]), h1 = bf2f(raw[CC + ch]), h2 = bf2f(raw[2 * CC + ch]);
        for (int r0 = 0; r0 < CH; r0 += 8) {
            float xs8[8], ob[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) xs8[u] = bf2f(raw[(r0 + u + 3) * CC + ch]);  // all taps before any store
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const float x = xs8[u];
                float out = fmaf(w.w, x, fmaf(w.z, h2, fmaf(w.y, h1, w.x * h0)));
                if (a.silu) out = __fdividef(out, 1.f + __expf(-out));
                ob[u] = (r0 + u < ntok) ? out : 0.f;
                h0 = h1;
                h1 = h2;
                h2 = x;
            }
            if (ch < D) {
#pragma unroll
                for (int u = 0; u < 8; ++u) qh[(r0 + u) * D + ch] = ob[u];
            } else if (ch < 2 * D) {
#pragma unroll
                for (int u = 0; u < 8; ++u) kh[(r0 + u) * D + ch - D] = ob[u];
            } else {
                umma::st_tf32x4(Vt, D, ch - 2 * D, r0, ob[0], ob[1], ob[2], ob[3]);
                umma::st_tf32x4(Vt, D, ch - 2 * D, r0 + 4, ob[4], ob[5], ob[6], ob[7]);
            }
        }
    }
    __syncthreads();
    // raw rows of positions pend-3 .. pend-1 (the conv window after this chunk), kept past P2
    uint4 *wstash = reinterpret_cast<uint4 *>(sm + I_MISC + 3200);
    if (tid < 3 * CC / 8) wstash[tid] = reinterpret_cast<const uint4 *>(raw + ntok * CC)[tid];
    for (int r = warp; r < ntok; r += NTI / 32) {
        const float nq = warp_dot_array(qh + r * D, qh + r * D, D);
        const float nk = warp_dot_array(kh + r * D, kh + r * D, D);
        const float rq = rsqrtf(nq + a.l2_eps), rk = rsqrtf(nk + a.l2_eps);
        for (int i = lane; i < D; i += 32) {
            qh[r * D + i] *= rq;
            kh[r * D + i] *= rk;
        }
    }
    {   // cumulative log decay along the chunk: 4 threads per channel, 16 tokens each
        const int ch = tid & 127, qd = tid >> 7;
        float acc = 0.f;
        for (int r = 16 * qd; r < 16 * qd + 16; ++r) {
            acc += G[r * D + ch];
            G[r * D + ch] = acc;
        }
        gtot[qd * D + ch] = acc;
        __syncthreads();
        float off = 0.f;
        for (int q2 = 0; q2 < qd; ++q2) off += gtot[q2 * D + ch];
        if (qd > 0)
            for (int r = 16 * qd; r < 16 * qd + 16; ++r) G[r * D + ch] += off;
    }
    __syncthreads();

    // ---- P2: [K+;Q+] and K- with a mid-chunk reference; Q+ tile to the workspace ----
    constexpr int MID = CH / 2;
    bool wide = false;
    if (tid < D) {
        const float g0 = G[tid], gm = G[MID * D + tid], gl = G[(CH - 1) * D + tid];
        wide = (g0 - gm > kMidRange) || (gm - gl > kMidRange);
        eGm[tid] = expf(gm);
        reinterpret_cast<float *>(blk + WS_GL)[tid] = expf(gl);
    }
    const bool slow = __syncthreads_or(wide) != 0;
    uint8_t *X1 = sm + I_X1;
    uint8_t *Km = sm + I_KM;
    for (int idx = tid; idx < CH * 16; idx += NTI) {
        const int r = idx >> 4, i0 = (idx & 15) * 8;  // 8 channels per item
        float xk[8], xq[8], xm[8], xp[8], gv[8], kv[8], qv[8], gmv[8], egv[8];
        *reinterpret_cast<float4 *>(gv) = *reinterpret_cast<const float4 *>(G + r * D + i0);
        *reinterpret_cast<float4 *>(gv + 4) = *reinterpret_cast<const float4 *>(G + r * D + i0 + 4);
        *reinterpret_cast<float4 *>(kv) = *reinterpret_cast<const float4 *>(kh + r * D + i0);
        *reinterpret_cast<float4 *>(kv + 4) = *reinterpret_cast<const float4 *>(kh + r * D + i0 + 4);
        *reinterpret_cast<float4 *>(qv) = *reinterpret_cast<const float4 *>(qh + r * D + i0);
        *reinterpret_cast<float4 *>(qv + 4) = *reinterpret_cast<const float4 *>(qh + r * D + i0 + 4);
        *reinterpret_cast<float4 *>(gmv) = *reinterpret_cast<const float4 *>(G + MID * D + i0);
        *reinterpret_cast<float4 *>(gmv + 4) = *reinterpret_cast<const float4 *>(G + MID * D + i0 + 4);
        *reinterpret_cast<float4 *>(egv) = *reinterpret_cast<const float4 *>(eGm + i0);
        *reinterpret_cast<float4 *>(egv + 4) = *reinterpret_cast<const float4 *>(eGm + i0 + 4);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const float g = gv[u], k_ = kv[u], q_ = qv[u];
            float eq;
            if (!slow) {
                const float ep = __expf(g - gmv[u]);
                xk[u] = k_ * ep;
                xq[u] = q_ * ep;
                xm[u] = k_ * __expf(gmv[u] - g);
                eq = ep * egv[u];
            } else {
                eq = __expf(g);
            }
            xp[u] = a.scale * q_ * eq;
        }
        if (!slow) {
            umma::st_bf16x8(X1, 128, r, i0, xk);
            umma::st_bf16x8(X1, 128, CH + r, i0, xq);
            umma::st_bf16x8(Km, CH, r, i0, xm);
        }
        umma::st_bf16x8(blk + WS_QP, CH, r, i0, xp);
    }
    fence_proxy_async_smem();
    umma::fence_before();
    __syncthreads();
    umma::fence_after();
    const uint32_t tmem = *tmem_s;
    uint32_t phase = 0;
    bool ok = true;
    if (!slow) {
        if (tid == 0) {
            const uint32_t id = umma::idesc(umma::kBF16, 128, CH);
            for (int ks = 0; ks < D / 16; ++ks)
                umma::mma_bf16(tmem, umma::sdesc_k(X1, 128, ks), umma::sdesc_k(Km, CH, ks), id, ks > 0);
            umma::commit(bar);
        }
        ok = wait_all(bar, phase);
        phase ^= 1;
        umma::fence_after();
    }
    // ---- P3: A (strict lower, fp32 in smem) and Qk (scaled, lower with diagonal, bf16 tile) ----
    float *A = reinterpret_cast<float *>(sm + I_A);      // [64][AST]
    float *Inv = reinterpret_cast<float *>(sm + I_INV);  // [64][64]
    // Qk tile staging: over q^ (dead) on the fast path; the slow path still reads q^, so it stages behind A
    uint8_t *Qks = slow ? sm + I_QKS_SLOW : sm + I_Q;
    if (ok && !slow) {
        float v[32];
        const int quad = warp & 3, half = (warp >> 2) & 1;  // warps 0-7: lanes 32*quad.., columns 32*half..
        if (warp < 8) umma::ld32(tmem + ((uint32_t)(32 * quad) << 16) + 32 * half, v);
        __syncthreads();  // every warp has read D1 and X1 is no longer read: A may overwrite it
        if (warp < 8) {
            const int row = 32 * quad + lane;
            if (row < CH) {
#pragma unroll
                for (int t = 0; t < 32; t += 4) {
                    const int s_ = 32 * half + t;
                    *reinterpret_cast<float4 *>(A + row * AST + s_) =
                        make_float4(s_ < row ? v[t] : 0.f, s_ + 1 < row ? v[t + 1] : 0.f, s_ + 2 < row ? v[t + 2] : 0.f,
                                    s_ + 3 < row ? v[t + 3] : 0.f);
                }
            } else {
                const int r = row - CH;
#pragma unroll
                for (int t = 0; t < 32; t += 8) {
                    float x8[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) x8[u] = (32 * half + t + u <= r) ? a.scale * v[t + u] : 0.f;
                    umma::st_bf16x8(Qks, CH, r, 32 * half + t, x8);
                }
            }
        }
    } else if (ok) {
        // decay range too wide for one reference point: exact pairwise exponentials
        for (int idx = tid; idx < CH * CH; idx += NTI) {
            const int r = idx / CH, s_ = idx - (idx / CH) * CH;
            float accA = 0.f, accQ = 0.f;
            if (s_ <= r && r < ntok) {
                for (int i = 0; i < D; ++i) {
                    const float ks = kh[s_ * D + i] * __expf(G[r * D + i] - G[s_ * D + i]);
                    accA = fmaf(kh[r * D + i], ks, accA);
                    accQ = fmaf(qh[r * D + i], ks, accQ);
                }
            }
            A[r * AST + s_] = s_ < r ? accA : 0.f;
            umma::st_bf16(Qks, CH, r, s_, s_ <= r ? a.scale * accQ : 0.f);
        }
    }
    if (__syncthreads_or(!ok)) {
        if (tid == 0) set_status(a.status, KDA_DEV_TIMEOUT);
        if (warp == 0) umma::dealloc(tmem, 256);
        return;
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {  // Qk tile to the workspace; the staging is reused by P4, so wait until it has been read
        bulk_s2g(blk + WS_QK, Qks, CH * CH * 2);
        bulk_commit();
        bulk_wait_read_all();
    }
    __syncthreads();
    // ---- P4: T = (I + diag(beta) A)^{-1} diag(beta), blocked by 16 ----
    // L = I + diag(beta) A; Inv = L^{-1}.  Diagonal 16x16 blocks by substitution, one column per thread.
    if (tid < CH) {
        const int b = tid >> 4, col = tid & 15, base = 16 * b;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            float acc = (r == col) ? 1.f : 0.f;
            const float br = beta[base + r];
#pragma unroll
            for (int s_ = 0; s_ < r; ++s_) acc = fmaf(-br * A[(base + r) * AST + base + s_], x[s_], acc);
            x[r] = acc;
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) Inv[(base + r) * CH + base + col] = x[r];
    }
    for (int idx = tid; idx < CH * CH; idx += NTI) {
        const int r = idx / CH, s_ = idx - (idx / CH) * CH;
        if ((s_ >> 4) > (r >> 4)) Inv[idx] = 0.f;
    }
    __syncthreads();
    float *P = reinterpret_cast<float *>(sm + I_T);  // [3][16][16] temporaries (K- is dead)
    for (int d = 1; d < 4; ++d) {
        const int nb = 4 - d;  // blocks (i, i-d) for i = d..3
        for (int idx = tid; idx < nb * 256; idx += NTI) {  // P_i = sum_{k=i-d}^{i-1} L_ik Inv_k,(i-d)
            const int bi = idx >> 8, rr = (idx >> 4) & 15, cc = idx & 15;
            const int i = bi + d, j = i - d;
            float acc = 0.f;
            for (int k = j; k < i; ++k)
#pragma unroll
                for (int t = 0; t < 16; ++t)
                    acc = fmaf(A[(16 * i + rr) * AST + 16 * k + t], Inv[(16 * k + t) * CH + 16 * j + cc], acc);
            P[idx] = beta[16 * i + rr] * acc;
        }
        __syncthreads();
        for (int idx = tid; idx < nb * 256; idx += NTI) {  // Inv_ij = -Inv_ii P_i
            const int bi = idx >> 8, rr = (idx >> 4) & 15, cc = idx & 15;
            const int i = bi + d, j = i - d;
            float acc = 0.f;
#pragma unroll
            for (int t = 0; t < 16; ++t) acc = fmaf(Inv[(16 * i + rr) * CH + 16 * i + t], P[bi * 256 + t * 16 + cc], acc);
            Inv[(16 * i + rr) * CH + 16 * j + cc] = -acc;
        }
        __syncthreads();
    }
    uint8_t *Tt = sm + I_T;  // T tf32 [64 r][64 s]: the B operand of W^T = K+^T T^T (K-major: row r, K = s)
    for (int idx = tid; idx < CH * 16; idx += NTI) {
        const int r = idx >> 4, s0 = (idx & 15) * 4;
        const float4 iv = *reinterpret_cast<const float4 *>(Inv + r * CH + s0);
        umma::st_tf32x4(Tt, CH, r, s0, iv.x * beta[s0], iv.y * beta[s0 + 1], iv.z * beta[s0 + 2], iv.w * beta[s0 + 3]);
    }
    __syncthreads();  // A / Inv are dead: Ktil^T may be staged over them
    // ---- P5: (k exp G)^T tile (A operand) and the Ktil^T workspace tile, 4 tokens per item ----
    uint8_t *Kpt = sm + I_Q;
    uint8_t *Kts = sm + I_A;
    for (int idx = tid; idx < D * 16; idx += NTI) {
        const int i = idx & 127, r0 = (idx >> 7) * 4;
        const float glast = G[(CH - 1) * D + i];
        float kp[4], kt[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float g = G[(r0 + u) * D + i], k_ = kh[(r0 + u) * D + i];
            kp[u] = k_ * __expf(g);
            kt[u] = k_ * __expf(glast - g);
        }
        umma::st_tf32x4(Kpt, D, i, r0, kp[0], kp[1], kp[2], kp[3]);
        umma::st_tf32x4(Kts, D, i, r0, kt[0], kt[1], kt[2], kt[3]);
    }
    fence_proxy_async_smem();
    umma::fence_before();
    __syncthreads();
    umma::fence_after();
    if (tid == 0) {
        const uint32_t id = umma::idesc(umma::kTF32, 128, CH);
        for (int ks = 0; ks < CH / 8; ++ks) {
            const uint64_t bt = umma::sdesc_k(Tt, CH, ks);
            umma::mma_tf32(tmem + 64, umma::sdesc_k(Kpt, D, ks), bt, id, ks > 0);
            umma::mma_tf32(tmem + 128, umma::sdesc_k(Vt, D, ks), bt, id, ks > 0);
        }
        umma::commit(bar);
    }
    if (tid == 0) {  // Ktil^T tile to the workspace (its staging is not reused)
        bulk_s2g(blk + WS_KT, Kts, D * CH * 4);
        bulk_commit();
    }
    ok = wait_all(bar, phase);
    phase ^= 1;
    umma::fence_after();
    if (!ok) {
        if (tid == 0) {
            set_status(a.status, KDA_DEV_TIMEOUT);
            bulk_wait_all();  // the Ktil^T copy still reads this CTA's shared memory
        }
        __syncthreads();
        if (warp == 0) umma::dealloc(tmem, 256);
        return;
    }
    // ---- P6: -W (bf16 tile [64 r][128 i]) and U' (fp32 [64 r][128 j]) via smem staging ----
    uint8_t *Wst = sm + I_K;
    float *Ust = reinterpret_cast<float *>(sm + I_G);
    if (warp < 8) {
        const int quad = warp & 3, half = warp >> 2;
        const int row = 32 * quad + lane;  // channel i (for W^T) / j (for U'^T)
        float v[32];
        umma::ld32(tmem + ((uint32_t)(32 * quad) << 16) + 64 + 32 * half, v);
#pragma unroll
        for (int t = 0; t < 32; ++t) umma::st_bf16(Wst, CH, 32 * half + t, row, -v[t]);
        umma::ld32(tmem + ((uint32_t)(32 * quad) << 16) + 128 + 32 * half, v);
#pragma unroll
        for (int t = 0; t < 32; ++t) Ust[(32 * half + t) * D + row] = v[t];
    }
    fence_proxy_async_smem();
    umma::fence_before();
    __syncthreads();
    if (tid == 0) {  // -W and U' to the workspace; every bulk copy of this CTA completes before it exits
        bulk_s2g(blk + WS_W, Wst, CH * D * 2);
        bulk_s2g(blk + WS_UP, Ust, CH * D * 4);
        bulk_commit();
        bulk_wait_all();
    }
    if (warp == 0) umma::dealloc(tmem, 256);

    // raw conv windows at a checkpoint boundary / at the sequence end (as the SIMT path)
    const int32_t flag = wsp<int32_t>(a, L.off_flags)[n];
    const int64_t pend = p0 + ntok;
    int wslot[2] = {-1, -1};
    if (a.interval > 0 && pend % a.interval == 0 && !(flag & kSeqCkptBad)) {
        const int64_t jj = pend / a.interval - start / a.interval - 1;
        const int s_ = a.ckpt_slots[a.ckpt_offsets[n] + jj];
        if (s_ >= a.num_slots || s_ < -1) {
            if (tid == 0) set_status(a.status, KDA_DEV_BAD_SLOT);
        } else {
            wslot[0] = s_;
        }
    }
    if (pend == start + len) wslot[1] = a.dst[n];
    for (int w = 0; w < 2; ++w) {
        if (wslot[w] < 0) continue;
        uint4 *cw = reinterpret_cast<uint4 *>(a.conv + ((size_t)wslot[w] * H + h) * (kConvW - 1) * CC);
        if (tid < 3 * CC / 8) cw[tid] = wstash[tid];
    }
}

}  // namespace tc

namespace tc {

// State kernel smem (bytes, from a 1024-aligned base)
constexpr uint32_t S_ST = 0;          // S^T bf16 tile [128 j][128 i]: A operand of U^T += S^T (-W)^T, O^T = S^T Q+^T
constexpr uint32_t S_OPS = 32768;     // one chunk's workspace block (Qk, -W, Q+, Ktil^T, gl, U'), WS_BLOCK bytes
constexpr uint32_t S_UT32 = 140288;   // U^T tf32 tile [128 j][64 r]: A operand of S^T += U^T Ktil
constexpr uint32_t S_UT16 = 173056;   // U^T bf16 tile [128 j][64 r]: A operand of O^T += U^T Qk^T
constexpr uint32_t S_OST = 189440;    // O staging fp32 [64 r][OST] (row stride 132: 16-byte rows, conflict-free)
constexpr int OST = 132;
constexpr uint32_t S_NW = 223232;     // RMSNorm weight [128]
constexpr uint32_t S_MISC = 223744;   // barriers, tensor-memory address
constexpr uint32_t S_SMEM = S_MISC + 256 + 1024;
static_assert(S_OPS + WS_BLOCK <= S_UT32 && S_UT32 % 1024 == 0 && S_UT16 % 1024 == 0, "state smem layout");
static_assert(S_OST + CH * OST * 4 <= S_NW, "state smem layout");

// TMEM columns: S^T [0,128), U^T [128,192), O^T [192,256)
constexpr uint32_t T_S = 0, T_U = 128, T_O = 192;

__global__ void __launch_bounds__(NT, 1) prefill_state_tc_kernel(const PrefillArgs a, const Layout2 L) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int H = a.H, CC = 3 * D;
    const int n = blockIdx.x, h = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int32_t flag = wsp<int32_t>(a, L.off_flags)[n];
    if (flag & kSeqInvalid) return;
    const int src = a.src[n], dst = a.dst[n];  // validated by the table kernel
    const int quad = warp & 3, half = warp >> 2;
    const int j = 32 * quad + lane;            // this thread's value channel = tensor-memory lane
    const uint32_t lane_off = (uint32_t)(32 * quad) << 16;
    uint8_t *Sst = sm + S_ST;
    uint8_t *ops = sm + S_OPS;
    uint8_t *Ut32 = sm + S_UT32;
    uint8_t *Ut16 = sm + S_UT16;
    float *Ost = reinterpret_cast<float *>(sm + S_OST);
    float *nw = reinterpret_cast<float *>(sm + S_NW);
    uint64_t *bar_ops = reinterpret_cast<uint64_t *>(sm + S_MISC);
    uint64_t *bar_mma = bar_ops + 1;
    uint32_t *tmem_s = reinterpret_cast<uint32_t *>(sm + S_MISC + 64);
    const int64_t start = a.start_pos[n];
    const int32_t c0 = wsp<int32_t>(a, L.off_seqc)[n], c1 = wsp<int32_t>(a, L.off_seqc)[n + 1];
    const ChunkEnt *ent = wsp<ChunkEnt>(a, L.off_ent);
    const int64_t *pos = wsp<int64_t>(a, L.off_pos);
    const uint8_t *blk0 = reinterpret_cast<const uint8_t *>(a.ws) + L.off_blk;
    auto blk_of = [&](int32_t c) { return blk0 + ((size_t)c * H + h) * WS_BLOCK; };

    if (warp == 0) umma::alloc(tmem_s, 256);
    for (int jj = tid; jj < D; jj += NT) nw[jj] = __ldg(a.norm_w + jj);
    if (tid == 0) {
        mbar_init(bar_ops, 1);
        mbar_init(bar_mma, 1);
        fence_mbar_init();
        if (c0 < c1) {
            mbar_arrive_expect_tx(bar_ops, WS_BLOCK);
            bulk_g2s(ops, blk_of(c0), WS_BLOCK, bar_ops);
        }
    }
    umma::fence_before();
    __syncthreads();
    umma::fence_after();
    const uint32_t tmem = *tmem_s;

    // initial state: S^T in tensor memory (lane j, column i) and its bf16 operand tile
    {
        float v[32];
        for (int part = 0; part < 2; ++part) {
            const int i0 = 64 * half + 32 * part;
#pragma unroll
            for (int t = 0; t < 32; ++t)
                v[t] = src >= 0 ? load_state(a.S, a.state_bf16, (((size_t)src * H + h) * D + i0 + t) * D + j) : 0.f;
            umma::st32(tmem + lane_off + T_S + i0, v);
#pragma unroll
            for (int t = 0; t < 32; t += 8) umma::st_bf16x8(Sst, D, j, i0 + t, v + t);
        }
    }
    uint32_t ph_ops = 0, ph_mma = 0;
    bool ok = true;
    for (int32_t c = c0; c < c1 && ok; ++c) {
        const ChunkEnt e = ent[c];
        const int64_t pend = pos[c] + e.n;
        int ck = -1;  // checkpoint slot of this chunk's end (looked up early; used after the state update)
        if (a.interval > 0 && pend % a.interval == 0 && !(flag & kSeqCkptBad)) {
            const int64_t jj = pend / a.interval - start / a.interval - 1;
            const int s_ = a.ckpt_slots[a.ckpt_offsets[n] + jj];
            if (s_ >= 0 && s_ < a.num_slots) ck = s_;
        }
        // the output gate of this warp's tokens (warp + 8k), channels 4*lane .. 4*lane+3, fetched early
        uint2 zr[8];
#pragma unroll
        for (int k8 = 0; k8 < 8; ++k8) {
            const int r = warp + 8 * k8;
            zr[k8] = (a.z && r < e.n)
                         ? __ldg(reinterpret_cast<const uint2 *>(a.z + ((size_t)(e.t0 + r) * H + h) * D) + lane)
                         : make_uint2(0u, 0u);
        }
        ok = mbar_wait(bar_ops, ph_ops);
        ph_ops ^= 1;
        // U' -> U^T columns of tensor memory (lane j, column r)
        if (ok) {
            float v[32];
            const float *up = reinterpret_cast<const float *>(ops + WS_UP);
#pragma unroll
            for (int t = 0; t < 32; ++t) v[t] = up[(32 * half + t) * D + j];
            umma::st32(tmem + lane_off + T_U + 32 * half, v);
        }
        fence_proxy_async_smem();
        umma::fence_before();
        __syncthreads();
        umma::fence_after();
        if (tid == 0 && ok) {
            const uint32_t idp = umma::idesc(umma::kBF16, 128, CH);
            for (int ks = 0; ks < D / 16; ++ks) {
                const uint64_t as = umma::sdesc_k(Sst, D, ks);
                umma::mma_bf16(tmem + T_U, as, umma::sdesc_k(ops + WS_W, CH, ks), idp, true);   // U^T += S^T (-W)^T
                umma::mma_bf16(tmem + T_O, as, umma::sdesc_k(ops + WS_QP, CH, ks), idp, ks > 0); // O^T = S^T Q+^T
            }
            umma::commit(bar_mma);
        }
        ok = __syncthreads_or(!ok) == 0 && wait_all(bar_mma, ph_mma);
        ph_mma ^= 1;
        umma::fence_after();
        if (!ok) break;
        // U^T -> its tf32 and bf16 operand tiles; decay the state columns by exp(G_last)
        {
            float v[32];
            umma::ld32(tmem + lane_off + T_U + 32 * half, v);
#pragma unroll
            for (int t = 0; t < 32; t += 4) umma::st_tf32x4(Ut32, D, j, 32 * half + t, v[t], v[t + 1], v[t + 2], v[t + 3]);
#pragma unroll
            for (int t = 0; t < 32; t += 8) umma::st_bf16x8(Ut16, D, j, 32 * half + t, v + t);
            const float *gl = reinterpret_cast<const float *>(ops + WS_GL);
            for (int part = 0; part < 2; ++part) {
                const int i0 = 64 * half + 32 * part;
                umma::ld32(tmem + lane_off + T_S + i0, v);
#pragma unroll
                for (int t = 0; t < 32; ++t) v[t] *= gl[i0 + t];
                umma::st32(tmem + lane_off + T_S + i0, v);
            }
        }
        fence_proxy_async_smem();
        umma::fence_before();
        __syncthreads();
        umma::fence_after();
        if (tid == 0) {
            const uint32_t ido = umma::idesc(umma::kBF16, 128, CH);
            for (int ks = 0; ks < CH / 16; ++ks)  // O^T += U^T Qk^T
                umma::mma_bf16(tmem + T_O, umma::sdesc_k(Ut16, D, ks), umma::sdesc_k(ops + WS_QK, CH, ks), ido, true);
            const uint32_t ids = umma::idesc(umma::kTF32, 128, D);
            for (int ks = 0; ks < CH / 8; ++ks)   // S^T += U^T Ktil
                umma::mma_tf32(tmem + T_S, umma::sdesc_k(Ut32, D, ks), umma::sdesc_k(ops + WS_KT, D, ks), ids, true);
            umma::commit(bar_mma);
        }
        ok = wait_all(bar_mma, ph_mma);
        ph_mma ^= 1;
        umma::fence_after();
        if (!ok) break;
        // the operand buffer is free: start the next chunk's copy
        if (tid == 0 && c + 1 < c1) {
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(bar_ops, WS_BLOCK);
            bulk_g2s(ops, blk_of(c + 1), WS_BLOCK, bar_ops);
        }
        // outputs: O^T -> staging -> gated RMSNorm -> y
        {
            float v[32];
            umma::ld32(tmem + lane_off + T_O + 32 * half, v);
#pragma unroll
            for (int t = 0; t < 32; ++t) Ost[(32 * half + t) * OST + j] = v[t];
        }
        __syncthreads();
#pragma unroll
        for (int k8 = 0; k8 < 8; ++k8) {  // one warp per token, 4 contiguous channels per lane
            const int r = warp + 8 * k8;
            const float4 o4 = *reinterpret_cast<const float4 *>(Ost + r * OST + 4 * lane);
            float ss = o4.x * o4.x;
            ss = fmaf(o4.y, o4.y, ss);
            ss = fmaf(o4.z, o4.z, ss);
            ss = fmaf(o4.w, o4.w, ss);
            ss = warp_sum(ss);
            const float rr = rsqrtf(ss * (1.0f / D) + a.rms_eps);
            if (r < e.n) {
                const float4 w4 = *reinterpret_cast<const float4 *>(nw + 4 * lane);
                float y0 = o4.x * rr * w4.x, y1 = o4.y * rr * w4.y, y2 = o4.z * rr * w4.z, y3 = o4.w * rr * w4.w;
                if (a.z) {
                    y0 *= sigmoid_gate(bf2f((uint16_t)(zr[k8].x & 0xffff)));
                    y1 *= sigmoid_gate(bf2f((uint16_t)(zr[k8].x >> 16)));
                    y2 *= sigmoid_gate(bf2f((uint16_t)(zr[k8].y & 0xffff)));
                    y3 *= sigmoid_gate(bf2f((uint16_t)(zr[k8].y >> 16)));
                }
                *(reinterpret_cast<uint2 *>(a.y + ((size_t)(e.t0 + r) * H + h) * D) + lane) =
                    make_uint2((uint32_t)f2bf(y0) | ((uint32_t)f2bf(y1) << 16),
                               (uint32_t)f2bf(y2) | ((uint32_t)f2bf(y3) << 16));
            }
        }
        // new state: bf16 operand tile for the next chunk; checkpoint when this chunk ends on a boundary
        {
            float v[32];
            for (int part = 0; part < 2; ++part) {
                const int i0 = 64 * half + 32 * part;
                umma::ld32(tmem + lane_off + T_S + i0, v);
#pragma unroll
                for (int t = 0; t < 32; t += 8) umma::st_bf16x8(Sst, D, j, i0 + t, v + t);
                if (ck >= 0) {
#pragma unroll
                    for (int t = 0; t < 32; ++t)
                        store_state(a.S, a.state_bf16, (((size_t)ck * H + h) * D + i0 + t) * D + j, v[t]);
                }
            }
        }
        __syncthreads();  // staging and tiles are reused by the next chunk
    }
    if (!ok) {
        if (tid == 0) set_status(a.status, KDA_DEV_TIMEOUT);
    } else {
        float v[32];
        for (int part = 0; part < 2; ++part) {
            const int i0 = 64 * half + 32 * part;
            umma::ld32(tmem + lane_off + T_S + i0, v);
#pragma unroll
            for (int t = 0; t < 32; ++t)
                store_state(a.S, a.state_bf16, (((size_t)dst * H + h) * D + i0 + t) * D + j, v[t]);
        }
        if (c0 == c1) {  // empty sequence: the window passes through unchanged
            uint16_t *cw = a.conv + ((size_t)dst * H + h) * (kConvW - 1) * CC;
            for (int idx = tid; idx < (kConvW - 1) * CC; idx += NT)
                cw[idx] = src >= 0 ? a.conv[((size_t)src * H + h) * (kConvW - 1) * CC + idx] : (uint16_t)0;
        }
    }
    umma::fence_before();
    __syncthreads();
    if (warp == 0) umma::dealloc(tmem, 256);
}

}  // namespace tc

}  // namespace

bool prefill_supported(int dk, int dv, int W, int chunk) {
    if (W != kConvW || (chunk != 16 && chunk != 64)) return false;
    return decode_supported(dk, dv, W);
}

static bool use_tensor_cores(int dk, int dv, int chunk) { return dk == 128 && dv == 128 && chunk == 64; }

size_t prefill_workspace_bytes(int H, int dk, int dv, int nseq, int64_t total_tokens, int chunk) {
    if (use_tensor_cores(dk, dv, chunk)) return tc::make_layout2(H, nseq, total_tokens).total;
    return make_layout(H, dk, dv, nseq, total_tokens, chunk).total;
}

static int launch_prefill_tc(const PrefillArgs &a, cudaStream_t st) {
    const tc::Layout2 L2 = tc::make_layout2(a.H, a.nseq, a.total_tokens);
    static int attr_done[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return launch_result("prefill: cudaGetDevice");
    if (!attr_done[dev]) {
        if (cudaFuncSetAttribute(tc::prefill_intra_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 tc::I_SMEM) != cudaSuccess ||
            cudaFuncSetAttribute(tc::prefill_state_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 tc::S_SMEM) != cudaSuccess)
            return launch_result("prefill: cudaFuncSetAttribute");
        attr_done[dev] = 1;
    }
    if (L2.maxc > 0x7fffffffLL || a.H > 65535) return fail(KDA_ERR_INVALID_ARG, "prefill: grid too large");
    prefill_table_kernel<<<1, kMaxSeqThreads, 0, st>>>(a, tc::as_layout(L2));
    if (a.total_tokens > 0) {
        dim3 gi((unsigned)L2.maxc, a.H);
        tc::prefill_intra_tc_kernel<<<gi, tc::NTI, tc::I_SMEM, st>>>(a, L2);
    }
    dim3 gs(a.nseq, a.H);
    tc::prefill_state_tc_kernel<<<gs, tc::NT, tc::S_SMEM, st>>>(a, L2);
    return launch_result("prefill (tensor-core path) launch");
}

int launch_prefill(const PrefillArgs &a, int dk, int dv, cudaStream_t st) {
    if (use_tensor_cores(dk, dv, a.chunk)) return launch_prefill_tc(a, st);
    const Layout L = make_layout(a.H, dk, dv, a.nseq, a.total_tokens, a.chunk);
    const int C = a.chunk;
    const size_t smem_intra = sizeof(float) * (3 * C * dk + C * (dk + dv) + 2 * C * C + C);
    const int DVT = std::min(dv, 32);
    const size_t smem_state = sizeof(float) * (dk * DVT + 3 * C * dk + C * C + 2 * C * DVT + dk);
    static int attr_done[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return launch_result("prefill: cudaGetDevice");
    if (!attr_done[dev]) {
        const int max_smem = 227 * 1024;
        if (cudaFuncSetAttribute(prefill_intra_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem) !=
                cudaSuccess ||
            cudaFuncSetAttribute(prefill_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem) !=
                cudaSuccess)
            return launch_result("prefill: cudaFuncSetAttribute");
        attr_done[dev] = 1;
    }
    if (L.maxc > 0x7fffffffLL || a.H > 65535) return fail(KDA_ERR_INVALID_ARG, "prefill: grid too large");
    prefill_table_kernel<<<1, kMaxSeqThreads, 0, st>>>(a, L);
    if (a.total_tokens > 0) {
        dim3 gi((unsigned)L.maxc, a.H);
        prefill_intra_kernel<<<gi, kThreads, smem_intra, st>>>(a, L, dk, dv);
    }
    dim3 gs(a.nseq, a.H, dv / DVT);
    prefill_state_kernel<<<gs, kThreads, smem_state, st>>>(a, L, dk, dv, DVT);
    if (a.total_tokens > 0) {
        dim3 go((unsigned)L.maxc, a.H);
        prefill_out_kernel<<<go, kThreads, 0, st>>>(a, L, dv);
    }
    return launch_result("prefill launch");
}

}  // namespace kda
