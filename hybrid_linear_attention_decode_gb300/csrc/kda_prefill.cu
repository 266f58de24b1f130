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
        S[idx] = src >= 0 ? a.S[(((size_t)src * H + h) * dk + i) * dv + j0 + j] : 0.f;
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
                    a.S[(((size_t)s * H + h) * dk + i) * dv + j0 + jj] = S[idx];
                }
            }
        }
    }
    for (int idx = tid; idx < dk * DVT; idx += kThreads) {
        const int i = idx / DVT, j = idx - (idx / DVT) * DVT;
        a.S[(((size_t)dst * H + h) * dk + i) * dv + j0 + j] = S[idx];
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

}  // namespace

bool prefill_supported(int dk, int dv, int W, int chunk) {
    if (W != kConvW || (chunk != 16 && chunk != 64)) return false;
    return decode_supported(dk, dv, W);
}

size_t prefill_workspace_bytes(int H, int dk, int dv, int nseq, int64_t total_tokens, int chunk) {
    return make_layout(H, dk, dv, nseq, total_tokens, chunk).total;
}

int launch_prefill(const PrefillArgs &a, int dk, int dv, cudaStream_t st) {
    const Layout L = make_layout(a.H, dk, dv, a.nseq, a.total_tokens, a.chunk);
    const int C = a.chunk;
    const size_t smem_intra = sizeof(float) * (3 * C * dk + C * (dk + dv) + 2 * C * C + C);
    const int DVT = std::min(dv, 32);
    const size_t smem_state = sizeof(float) * (dk * DVT + 3 * C * dk + C * C + 2 * C * DVT + dk);
    static int attr_done[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return KDA_ERR_CUDA;
    if (!attr_done[dev]) {
        const int max_smem = 227 * 1024;
        if (cudaFuncSetAttribute(prefill_intra_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem) !=
                cudaSuccess ||
            cudaFuncSetAttribute(prefill_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem) !=
                cudaSuccess)
            return KDA_ERR_CUDA;
        attr_done[dev] = 1;
    }
    if (L.maxc > 0x7fffffffLL || a.H > 65535) return KDA_ERR_INVALID_ARG;
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
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // namespace kda
