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
// Two implementations, both graph-capturable:
//   * SIMT fp32, for every supported shape (chunk 16 or 64), four launches on the caller's stream:
//     1. table:  validates cu_seqlens / start_pos / checkpoint offsets, builds the chunk table;
//     2. intra:  one CTA per (chunk, head): causal conv + SiLU, L2 norms, gates, A, Qk, the unit-lower
//                triangular solve, W / U' / decayed K / decayed Q into the workspace; conv windows of
//                checkpoints and of the final state go straight to the pool;
//     3. state:  one CTA per (sequence, head, dv tile), sequential over the sequence's chunks: U, O and
//                the state chain in fp32; checkpoint states at every boundary, the final one to dst;
//     4. out:    gated RMSNorm of O into the bf16 output.
//   * tcgen05 (namespace tc), for dk = dv = 128 and chunk 64: the same table, then a persistent intra
//     kernel (one CTA per SM looping over (chunk, head) items, operand tiles written to the workspace in
//     their shared-memory layout) and a state kernel (one CTA per (sequence, head): the chunk chain with
//     S^T in tensor memory, the gated RMSNorm on separate warps beside it).  A long call with few
//     (sequence, head) chains is launched in segments, the state chain of one segment running on a side
//     stream beside the intra kernel of the next (launch_prefill_tc).
#include <cuda.h>  // CUtensorMap; the encoder is looked up at run time, so nothing links the driver library

#include <algorithm>
#include <atomic>
#include <mutex>

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

// Everything the tensor-core intra kernel needs to know about a chunk, written by the table kernel so that the
// kernel fetches it with one round of loads.
struct __align__(16) ItemMeta {
    int32_t seq, t0, n, srcv;    // sequence, first token, tokens, source slot
    int64_t p0, start, ts, len;  // first position, the sequence's start position, first token and length
};
static_assert(sizeof(ItemMeta) == 48, "three 16-byte words");

enum : int32_t { kSeqInvalid = 1, kSeqCkptBad = 2 };

struct Layout {
    int64_t maxc;
    size_t off_cnt, off_ent, off_pos, off_seqc, off_flags;
    size_t off_win;   // bf16 [nseq][H][W-1][2dk+dv]: the source slots' windows as they were when the call began
    int32_t win_u4;   // 16-byte words per (sequence, head) window
    size_t off_meta;  // ItemMeta [maxc] (tensor-core path), 0 when absent
    size_t off_W, off_U, off_Kt, off_Qp, off_Qk, off_gl, off_O;
    size_t total;
};

// 16-byte words of one stored conv window ([W-1][2dk+dv] bf16; a whole number of words for every supported
// shape, whose dk and dv are multiples of 16).
inline int32_t window_u4(int dk, int dv) { return (int32_t)((kConvW - 1) * (2 * dk + dv) * 2 / 16); }

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
    L.win_u4 = window_u4(dk, dv);
    L.off_win = o; o = align256(o + (size_t)16 * L.win_u4 * nseq * H);
    L.off_meta = 0;
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
// call's tokens when pos >= start, else from the source window as it was when the call began (`win`, the
// sequence's snapshot for this head; zeros for src = -1).
__device__ __forceinline__ uint16_t raw_at(const PrefillArgs &a, int dk, int dv, int h, int ch, int64_t pos,
                                           int64_t start, int64_t ts, int src, const uint16_t *win) {
    if (pos >= start) return raw_bits(a, dk, dv, ts + (pos - start), h, ch);
    if (src < 0) return 0;
    const int CC = 2 * dk + dv;
    const int row = (int)(pos - start + (kConvW - 1));
    return win[row * CC + ch];
}

// ------------------------------------------------------------------------------------------ 1. table
// Block 0 validates the tables and builds the chunk table.  The other blocks copy each sequence's source
// window (src >= 0) into the workspace: the intra kernels read a sequence's history rows from that copy,
// never from the pool, so an in-place call (src == dst) cannot see the destination window that the item of
// the sequence's last chunk writes, whichever CTA runs first.
__global__ void __launch_bounds__(kMaxSeqThreads) prefill_table_kernel(const PrefillArgs a, const Layout L) {
    __shared__ int32_t scan[kMaxSeqThreads];
    __shared__ int32_t carry_s;
    const int tid = threadIdx.x;
    if (blockIdx.x > 0) {
        const int64_t words = (int64_t)a.nseq * a.H * L.win_u4;
        uint4 *snap = wsp<uint4>(a, L.off_win);
        const uint4 *pool = reinterpret_cast<const uint4 *>(a.conv);
        for (int64_t w = (int64_t)(blockIdx.x - 1) * kMaxSeqThreads + tid; w < words;
             w += (int64_t)(gridDim.x - 1) * kMaxSeqThreads) {
            const int64_t unit = w / L.win_u4, n = unit / a.H;
            const int h = (int)(unit - n * a.H);
            const int src = a.src[n];
            if (src >= 0 && src < a.num_slots)  // range-checked here too: block 0 validates concurrently
                snap[w] = pool[((int64_t)src * a.H + h) * L.win_u4 + (w - unit * L.win_u4)];
        }
        return;
    }
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
        if (L.off_meta) {
            ItemMeta m;
            m.seq = n;
            m.t0 = e.t0;
            m.n = e.n;
            m.srcv = a.src[n];
            m.p0 = p0;
            m.start = start;
            m.ts = a.cu_seqlens[n];
            m.len = len;
            wsp<ItemMeta>(a, L.off_meta)[c] = m;
        }
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
    const uint16_t *win = wsp<uint16_t>(a, L.off_win) + ((size_t)n * H + h) * L.win_u4 * 8;

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
        for (int j = 0; j < kConvW - 1; ++j) hist[j] = bf2f(raw_at(a, dk, dv, h, ch, p0 - (kConvW - 1) + j, start, ts, srcv, win));
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
            cw[idx] = raw_at(a, dk, dv, h, ch, pend - (kConvW - 1) + row, start, ts, srcv, win);
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
//   [A ; Qk]  = [K+ ; Q+] (mid-chunk reference) x K-^T           tf32, M=128 N=64  K=128 (two halves)
//   W^T       = (k*exp(G))^T x T^T,   U'^T = V^T x T^T            tf32, M=128 N=64  K=64
//   U^T       = U'^T + S^T x (-W)^T                                bf16, M=128 N=64  K=128
//   O^T       = S^T x Q+^T                                         bf16, M=128 N=64  K=128
//             + U^T x Qk^T                                         tf32, M=128 N=64  K=64
//   S^T       = S^T Diag(exp(G_last)) + U^T x Ktil                 tf32, M=128 N=128 K=64
// tf32 operands are rounded to nearest (cvt.rna); accumulation is fp32 in tensor memory.  The diagonal of
// Qk is not taken from the MMA: it is scale * (q^_r . k^_r), summed in fp32 from the normalised vectors.
// Where q^_r and k^_r are nearly orthogonal (a sequence's first token from an empty state makes O_r that
// single term) the rounded operands of the MMA would lose the dot product's relative accuracy, and the
// gated RMSNorm scales the output back up to unit size.
namespace tc {

constexpr int D = 128, CH = 64;
constexpr float kMidRange = 40.f;  // |G_r - G_mid| bound for the factorised A / Qk (fp32-safe)

// Workspace block per (chunk, head); the first WS_OPS bytes are operand tiles in their shared-memory
// layout (K-major, 128B swizzle), copied verbatim by the state kernel.
constexpr uint32_t WS_QK = 0;                    // tf32 [64 r][64 s]    Qk (scaled, masked, fp32 diagonal)
constexpr uint32_t WS_W = WS_QK + CH * CH * 4;   // bf16 [64 r][128 i]   -W (negated)
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
    size_t off_cnt, off_ent, off_pos, off_seqc, off_flags, off_win, off_meta, off_blk, off_carry, total;
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
    L.off_win = o; o = align256(o + (size_t)16 * window_u4(D, D) * nseq * H);
    L.off_meta = o; o = align256(o + sizeof(ItemMeta) * L.maxc);
    o = (o + 1023) & ~size_t(1023);
    L.off_blk = o; o += (size_t)WS_BLOCK * L.maxc * H;
    L.off_carry = o; o += (size_t)nseq * H * D * D * 4;  // fp32 state of each (sequence, head) between segments
    L.total = o;
    return L;
}

inline Layout as_layout(const Layout2 &L2) {  // the table kernel only uses these fields
    Layout L{};
    L.maxc = L2.maxc;
    L.off_cnt = L2.off_cnt; L.off_ent = L2.off_ent; L.off_pos = L2.off_pos;
    L.off_seqc = L2.off_seqc; L.off_flags = L2.off_flags;
    L.off_win = L2.off_win; L.win_u4 = window_u4(D, D); L.off_meta = L2.off_meta;
    return L;
}

__device__ __forceinline__ bool wait_all(uint64_t *bar, uint32_t parity) {
    const bool ok = mbar_wait(bar, parity);
    return __syncthreads_or(!ok) == 0;
}

// Intra-chunk kernel smem (bytes, from a 1024-aligned base), by phase:
//   P0-P1  [0,32K) q^ fp32 | [32K,64K) k^ fp32 | [64K,96K) G fp32 (decay logits staged in its first 16K) |
//          [96K,128K) V^T tf32 tile | [128K,180K) raw rows
//   P2     [128K,160K) [K+;Q+] tf32 tile | [160K,176K) K- tf32 tile (one channel half at a time)
//   P2 also writes, on the fast path, fp32 K+ = k^ exp(G - G_mid) over k^ and K- = k^ exp(G_mid - G) over G
//   P3-P4  [188K,204K) Qk tf32 staging (its copy-out is read by the end of the item) | [0,17K) Inv fp32 (row
//          stride 68) | [128K,145K) A fp32 (row stride 68) | [160K,176K) block temps, then T tf32
//   P5     [0,32K) (k exp G)^T tf32 tile | [128K,160K) Ktil^T tf32 staging
//   P6     [32K,48K) -W bf16 staging | [96K,128K) U' fp32 staging (both copied out by the start of the next item)
constexpr uint32_t I_Q = 0, I_K = 32768, I_G = 65536, I_VT = 98304, I_RAW = 131072;
constexpr uint32_t I_X1 = 131072, I_KM = 163840, I_A = 131072, I_T = 163840;
constexpr uint32_t I_INV = 0;          // Inv fp32 [64][IST] over q^ (free after the Qk copy-out)
constexpr uint32_t I_MISC = 184320;   // beta, exp(G_mid), decay partial sums, barrier, tmem address, window stash,
                                      // fp32 q^.k^ per row, G_mid, exp(G_last - G_mid), G row 0
constexpr uint32_t I_QKS = 192512;    // Qk tf32 staging [64][64]
constexpr uint32_t I_SMEM = I_QKS + CH * CH * 4 + 1024;  // + alignment slack
constexpr int RAW_ROWS = CH + kConvW - 1;           // 3 history rows + 64 tokens
constexpr int AST = 68;                             // row stride of A in smem (padded against bank conflicts)
constexpr int IST = 68;                             // row stride of Inv in smem (the same padding)
static_assert(I_A + CH * AST * 4 <= I_T && I_MISC + 7424 <= I_QKS && I_QKS % 1024 == 0, "A, misc, Qk staging");
static_assert(I_RAW + RAW_ROWS * 3 * D * 2 <= I_MISC, "raw staging");
static_assert(I_INV + CH * IST * 4 <= I_K && (IST * 4) % 16 == 0, "Inv staging");

constexpr int NTI = 512;  // intra kernel threads
constexpr int RAW_PART = RAW_ROWS * D;  // elements of one raw block ([67][128] bf16 of q, k or v)
static_assert((RAW_PART * 2) % 128 == 0, "raw blocks stay 128-byte aligned");


// Tiled TMA load of a (channel, head, token) box of a [T][H][128] bf16 token tensor into shared memory,
// completion counted on `bar`.  The channel coordinate is always 0; token coordinates outside [0, T) read
// zeros.
__device__ __forceinline__ void tma_load_tokens(void *dst, const CUtensorMap *map, int head, int token,
                                                uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(head), "r"(token), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ float log_sigmoid_fast(float x) {
    // log(sigmoid(x)) = min(x, 0) - log(1 + exp(-|x|)); absolute error ~1e-7, which is what the
    // cumulative decay (a sum of these) needs
    return fminf(x, 0.f) - __logf(1.f + __expf(-fabsf(x)));
}

// Sums of NV values per lane over the 32 lanes of a warp by recursive halving (NV a power of two, 2..32): at each
// step a lane keeps half of its values, adds the partner's matching half, and passes the other half on.  Lane l
// returns the total of value l >> (5 - log2 NV); v is overwritten.
template <int NV>
__device__ __forceinline__ float warp_reduce_scatter(float *v, int lane) {
    static_assert(NV >= 2 && NV <= 32 && (NV & (NV - 1)) == 0, "a power of two");
#pragma unroll
    for (int n = NV, off = 16; n > 1; n >>= 1, off >>= 1) {
        const bool up = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            const float send = up ? v[i] : v[i + n / 2];
            const float keep = up ? v[i + n / 2] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
    }
    float r = v[0];
#pragma unroll
    for (int off = 32 / NV; off > 1; off >>= 1) r += __shfl_xor_sync(0xffffffffu, r, off >> 1);
    return r;
}

// Packed fp32 pairs (fma / mul / add .f32x2 round each lane as the scalar instruction would).
__device__ __forceinline__ uint64_t pk2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void upk2(uint64_t v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
constexpr float kLog2e = 1.4426950408889634f;
__device__ __forceinline__ float ex2_approx(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}
// two bf16 (low half first) as a packed fp32 pair
__device__ __forceinline__ uint64_t bf2x2(uint32_t w) { return pk2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u)); }
// x * sigmoid(x) of both lanes with one reciprocal: with y = 1 + exp(-x), 1/y0 = y1 / (y0 y1) and 1/y1 = y0 / (y0 y1).
// exp(-x) is capped at 2^57 (x below about -39.5, where x sigmoid(x) is below 1e-15 in magnitude) so that the
// product stays finite.
__device__ __forceinline__ uint64_t silu2(uint64_t x) {
    float t0, t1;
    upk2(mul2(x, pk2(-kLog2e, -kLog2e)), t0, t1);
    const float e0 = ex2_approx(fminf(t0, 57.f)), e1 = ex2_approx(fminf(t1, 57.f));
    float y0, y1;
    upk2(add2(pk2(e0, e1), pk2(1.f, 1.f)), y0, y1);
    float rp;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(rp) : "f"(y0 * y1));
    return mul2(x, pk2(rp * y1, rp * y0));
}

__global__ void __launch_bounds__(NTI, 1)
    prefill_intra_tc_kernel(const PrefillArgs a, const Layout2 L, const __grid_constant__ CUtensorMap tm_q,
                            const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                            const __grid_constant__ CUtensorMap tm_a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int H = a.H, CC = 3 * D;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // work items (chunk, head), head fastest: those of the chunks [seg_lo, seg_hi)
    const int item_lo = a.seg_lo * H;
    const int total = min(*wsp<int32_t>(a, L.off_cnt), a.seg_hi) * H;
    if (item_lo + (int)blockIdx.x >= total) return;

    float *qh = reinterpret_cast<float *>(sm + I_Q);
    float *kh = reinterpret_cast<float *>(sm + I_K);
    float *G = reinterpret_cast<float *>(sm + I_G);
    uint8_t *Vt = sm + I_VT;
    uint16_t *raw = reinterpret_cast<uint16_t *>(sm + I_RAW);  // q, k, v blocks [67][128] bf16, row = position p0-3+row
    uint16_t *astage = reinterpret_cast<uint16_t *>(sm + I_G);  // decay logits bf16 [64][128] (G comes later)
    float *beta = reinterpret_cast<float *>(sm + I_MISC);
    float *eGm = beta + 64;     // exp(G_mid) per channel
    float *gtot = eGm + D;      // [128] cumulative decay of tokens 0-31 (the decay sums)
    ItemMeta *meta = reinterpret_cast<ItemMeta *>(sm + I_MISC + 2816);  // [2], by item parity
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + I_MISC + 3072);
    uint64_t *bar_in = bar + 1;
    uint32_t *tmem_s = reinterpret_cast<uint32_t *>(sm + I_MISC + 3136);
    uint4 *wstash = reinterpret_cast<uint4 *>(sm + I_MISC + 3200);  // raw rows of the window after the chunk
    float *qkd = reinterpret_cast<float *>(sm + I_MISC + 5632);      // [64] q^_r . k^_r in fp32
    float *gmid = reinterpret_cast<float *>(sm + I_MISC + 5888);     // [128] G_mid
    float *eglm = reinterpret_cast<float *>(sm + I_MISC + 6400);     // [128] exp(G_last - G_mid)
    float *g0s = reinterpret_cast<float *>(sm + I_MISC + 6912);      // [128] G row 0

    // Item metadata from global memory (one thread; dependent loads).
    // Item metadata: the table kernel's record of the item's chunk (one round of three 16-byte loads).
    auto load_meta = [&](int item, ItemMeta *m) {
        const uint4 *rec = reinterpret_cast<const uint4 *>(wsp<ItemMeta>(a, L.off_meta) + item / H);
        const uint4 r0 = __ldg(rec), r1 = __ldg(rec + 1), r2 = __ldg(rec + 2);
        uint4 *d = reinterpret_cast<uint4 *>(m);
        d[0] = r0;
        d[1] = r1;
        d[2] = r2;
    };
    // TMA loads of an item's rows: 67 token rows of q, k and v starting 3 tokens before the chunk (zeros
    // before the first token), and separately (its region frees later) the chunk's 64 rows of decay logits.
    // Both count on one phase of bar_in; rows past the chunk's last token hold whatever follows and every
    // use of them is masked.
    auto issue_rows = [&](const ItemMeta &m, int h) {
        mbar_arrive_expect_tx(bar_in, 3 * RAW_PART * 2 + CH * D * 2);
        tma_load_tokens(raw, &tm_q, h, m.t0 - (kConvW - 1), bar_in);
        tma_load_tokens(raw + RAW_PART, &tm_k, h, m.t0 - (kConvW - 1), bar_in);
        tma_load_tokens(raw + 2 * RAW_PART, &tm_v, h, m.t0 - (kConvW - 1), bar_in);
    };
    auto issue_logits = [&](const ItemMeta &m, int h) { tma_load_tokens(astage, &tm_a, h, m.t0, bar_in); };

    if (warp == 0) umma::alloc(tmem_s, 256);
    if (tid == 0) {
        mbar_init(bar, 1);
        mbar_init(bar_in, 1);
        fence_mbar_init();
        load_meta(item_lo + blockIdx.x, &meta[0]);
        issue_rows(meta[0], (item_lo + (int)blockIdx.x) % H);
        issue_logits(meta[0], (item_lo + (int)blockIdx.x) % H);
    }
    __syncthreads();  // barriers, the tensor-memory address and the first item's metadata are in place
    const uint32_t tmem = *tmem_s;
    uint32_t phase = 0, ph_in = 0;
    bool ok = true, in_flight = true;  // in_flight: row loads issued and not yet waited for (thread 0's view)
    // the first item's beta logit; later items get theirs prefetched by the item before
    uint16_t blogit = (tid < CH && tid < meta[0].n)
                          ? a.b[(size_t)(meta[0].t0 + tid) * H + (item_lo + (int)blockIdx.x) % H]
                          : (uint16_t)0;

    for (int item = item_lo + blockIdx.x, it = 0; item < total; item += gridDim.x, ++it) {
    const int c = item / H, h = item - (item / H) * H;
    const int next = item + gridDim.x;
    const bool has_next = next < total;
    const int ntok = meta[it & 1].n;
    uint8_t *blk = reinterpret_cast<uint8_t *>(a.ws) + L.off_blk + ((size_t)c * H + h) * WS_BLOCK;
    if (tid == 0) bulk_wait_read_all();  // the item before's -W and U' copy-outs: their staging is rewritten below
    float4 cw3[3][2];  // conv weights of this thread's three conv units (P1), in flight during the wait below
#pragma unroll
    for (int k = 0; k < 3; ++k) {
        const float4 *wp = reinterpret_cast<const float4 *>(a.conv_w + ((size_t)h * CC + 2 * ((tid + k * NTI) % (CC / 2))) * kConvW);
        cw3[k][0] = __ldg(wp);
        cw3[k][1] = __ldg(wp + 1);
    }
    ok = !__syncthreads_or(!mbar_wait(bar_in, ph_in));
    if (!ok) break;  // the loads stay in flight: the exit path waits for them once more
    ph_in ^= 1;
    if (tid == 0) in_flight = false;
    if (tid < CH) beta[tid] = tid < ntok ? sigmoidf_(bf2f(blogit)) : 0.f;  // read from P4 on
    {   // history rows before the sequence start: the source window as it was when the call began (the
        // table kernel's snapshot), or zeros.  Only an item that has such rows needs the barrier (the condition
        // is the same for every thread).
        const ItemMeta mt = meta[it & 1];
        const int hist_src = (int)min((int64_t)(kConvW - 1), max((int64_t)0, mt.start - mt.p0 + (kConvW - 1)));
        if (hist_src > 0) {
            const uint16_t *win = wsp<uint16_t>(a, L.off_win) + ((size_t)mt.seq * H + h) * (kConvW - 1) * CC;
            for (int idx = tid; idx < hist_src * CC; idx += NTI) {
                const int row = idx / CC, ch = idx - (idx / CC) * CC;
                const int64_t p = mt.p0 - (kConvW - 1) + row;
                raw[(ch >> 7) * RAW_PART + row * D + (ch & 127)] =
                    mt.srcv >= 0 ? win[(p - mt.start + (kConvW - 1)) * CC + ch] : (uint16_t)0;
            }
            __syncthreads();
        }
    }
    // ---- P1: causal conv + SiLU over (channel pair, block of 8 rows) units, three per thread, in packed fp32
    //      pairs: the block's three history rows come from the staged raw rows, the window runs in registers
    //      along the block.  A warp's 32 pairs are 64 channels of one of q, k, v. ----
    static_assert((CC / 2) * (CH / 8) == 3 * NTI && (CC / 2) % 32 == 0, "three conv units per thread");
#pragma unroll
    for (int k = 0; k < 3; ++k) {
        const int u = tid + k * NTI, cp = u % (CC / 2), rb = u / (CC / 2);
        const int part = cp >> 6, cc = 2 * cp - 128 * part, r0 = 8 * rb;
        const float4 wa = cw3[k][0], wb = cw3[k][1];  // taps of channels cc, cc + 1 (tap 3 on the current row)
        const uint64_t w0 = pk2(wa.x, wb.x), w1 = pk2(wa.y, wb.y), w2 = pk2(wa.z, wb.z), w3 = pk2(wa.w, wb.w);
        const uint32_t *rp = reinterpret_cast<const uint32_t *>(raw + part * RAW_PART + r0 * D + cc);  // row r0 = position r0 - 3
        uint64_t h0 = bf2x2(rp[0]), h1 = bf2x2(rp[D / 2]), h2 = bf2x2(rp[D]);
        uint64_t ob[8];
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) ob[kk] = bf2x2(rp[(kk + 3) * (D / 2)]);  // all rows before any store
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const uint64_t x = ob[kk];
            uint64_t out = fma2(w3, x, fma2(w2, h2, fma2(w1, h1, mul2(w0, h0))));
            ob[kk] = a.silu ? silu2(out) : out;
            h0 = h1;
            h1 = h2;
            h2 = x;
        }
        if (r0 + 8 > ntok) {  // the chunk ends inside this block (warp-uniform): rows past it are zero
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                if (r0 + kk >= ntok) ob[kk] = 0;
        }
        if (part < 2) {
            float *dstp = (part == 0 ? qh : kh) + r0 * D + cc;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) *reinterpret_cast<uint64_t *>(dstp + kk * D) = ob[kk];
        } else {
            float lo[8], hi[8];
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) upk2(ob[kk], lo[kk], hi[kk]);
            umma::st_tf32x4(Vt, D, cc, r0, lo[0], lo[1], lo[2], lo[3]);
            umma::st_tf32x4(Vt, D, cc, r0 + 4, lo[4], lo[5], lo[6], lo[7]);
            umma::st_tf32x4(Vt, D, cc + 1, r0, hi[0], hi[1], hi[2], hi[3]);
            umma::st_tf32x4(Vt, D, cc + 1, r0 + 4, hi[4], hi[5], hi[6], hi[7]);
        }
    }
    __syncthreads();
    // raw rows of positions pend-3 .. pend-1 (the conv window after this chunk), kept past P2
    if (tid < 3 * CC / 8) {  // [3][q|k|v] rows, the layout of a stored window
        const int r3 = tid / (CC / 8), rem = tid - r3 * (CC / 8), part = rem >> 4, unit = rem & 15;
        wstash[tid] = reinterpret_cast<const uint4 *>(raw + part * RAW_PART + (ntok + r3) * D)[unit];
    }
    {   // L2 norms of q and k rows 4 warp .. 4 warp + 3 (lane: channels 4 lane .. 4 lane + 3 of each), and q^.k^
        const int rw = 4 * warp;
        float4 vq[4], vk[4];
        float ss[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            vq[j] = *reinterpret_cast<const float4 *>(qh + (rw + j) * D + 4 * lane);
            vk[j] = *reinterpret_cast<const float4 *>(kh + (rw + j) * D + 4 * lane);
            ss[2 * j] = fmaf(vq[j].w, vq[j].w, fmaf(vq[j].z, vq[j].z, fmaf(vq[j].y, vq[j].y, vq[j].x * vq[j].x)));
            ss[2 * j + 1] = fmaf(vk[j].w, vk[j].w, fmaf(vk[j].z, vk[j].z, fmaf(vk[j].y, vk[j].y, vk[j].x * vk[j].x)));
        }
        const float rs = rsqrtf(warp_reduce_scatter<8>(ss, lane) + a.l2_eps);  // lane l: row l / 8, k if l % 8 >= 4
        float dq[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float rq = __shfl_sync(0xffffffffu, rs, 8 * j), rk = __shfl_sync(0xffffffffu, rs, 8 * j + 4);
            vq[j].x *= rq; vq[j].y *= rq; vq[j].z *= rq; vq[j].w *= rq;
            vk[j].x *= rk; vk[j].y *= rk; vk[j].z *= rk; vk[j].w *= rk;
            dq[j] = fmaf(vq[j].w, vk[j].w, fmaf(vq[j].z, vk[j].z, fmaf(vq[j].y, vk[j].y, vq[j].x * vk[j].x)));
            if (rw + j < ntok) {
                *reinterpret_cast<float4 *>(qh + (rw + j) * D + 4 * lane) = vq[j];
                *reinterpret_cast<float4 *>(kh + (rw + j) * D + 4 * lane) = vk[j];
            }
        }
        const float dqk = warp_reduce_scatter<4>(dq, lane);  // lane l: row l / 8
        if ((lane & 7) == 0) qkd[rw + (lane >> 3)] = rw + (lane >> 3) < ntok ? dqk : 0.f;
    }
    bool wide = false;
    {   // cumulative log decay along the chunk from the staged logits: 4 threads per channel, 16 tokens each,
        // in registers; G overwrites the staging only after every logit has been read
        const int ch = tid & 127, qd = tid >> 7;
        float g16[16];
        float acc = 0.f;
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const int r = 16 * qd + u;
            acc += r < ntok ? log_sigmoid_fast(bf2f(astage[r * D + ch])) : 0.f;
            g16[u] = acc;
        }
        gtot[qd * D + ch] = acc;
        if (qd == 0) g0s[ch] = g16[0];
        __syncthreads();
        float off = 0.f;
        for (int q2 = 0; q2 < qd; ++q2) off += gtot[q2 * D + ch];
#pragma unroll
        for (int u = 0; u < 16; ++u) G[(16 * qd + u) * D + ch] = qd > 0 ? g16[u] + off : g16[u];
        static_assert(CH / 2 == 32, "G_mid is the first row of the third quarter");
        if (qd == 2) {
            // the mid-chunk reference G_mid = G row 32 and G_last = G row 63 of this channel, each summed exactly
            // as its row of G is above, and whether the chunk's decay range is too wide for one reference
            const float gm = g16[0] + off, gl = gtot[3 * D + ch] + (off + gtot[2 * D + ch]);
            wide = (g0s[ch] - gm > kMidRange) || (gm - gl > kMidRange);
            eGm[ch] = expf(gm);
            gmid[ch] = gm;
            eglm[ch] = expf(gl - gm);
            reinterpret_cast<float *>(blk + WS_GL)[ch] = expf(gl);
        }
    }
    const bool slow = __syncthreads_or(wide) != 0;

    // ---- P2: [K+;Q+] and K- with a mid-chunk reference; Q+ tile to the workspace ----
    uint8_t *X1 = sm + I_X1;  // [K+; Q+] tf32 [128 rows][64 channels] of one channel half
    uint8_t *Km = sm + I_KM;  // K- tf32 [64 rows][64 channels] of one channel half
    {   // The [A; Qk] MMA takes tf32 operands and runs in two channel halves whose tiles take the space of one
        // bf16 tile over all channels.  The operands of half 1 are formed in registers while the MMAs of half
        // 0 run, and stored once those MMAs have read the tiles.  Rows warp + 16 j, two channels per thread
        // per half: the 8-byte reads of G, k^ and q^ are consecutive across a warp and each 8-byte tile store
        // fills a contiguous row chunk.
        const int c2 = 2 * lane;
        float xk[4][2], xq[4][2], xm[4][2];  // K+, Q+ (mid reference), K- of the thread's rows and channels
        auto form = [&](int hh) {  // ... of channel half hh; Q+ (chunk start) of that half to the workspace
            // (packed pairs of the thread's two channels: exp(G - G_mid) and exp(G_mid - G) share one argument)
            const int ic = 64 * hh + c2;
            const float2 m2 = *reinterpret_cast<const float2 *>(gmid + ic);  // (row 32 of G is overwritten below)
            const float2 e2 = *reinterpret_cast<const float2 *>(eGm + ic);
            const uint64_t ngm2 = pk2(-m2.x, -m2.y), eg2 = pk2(e2.x, e2.y);
            const uint64_t l2e2 = pk2(kLog2e, kLog2e), sc2 = pk2(a.scale, a.scale);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int r = warp + 16 * j;
                const uint64_t g2 = *reinterpret_cast<const uint64_t *>(G + r * D + ic);
                const uint64_t k2 = *reinterpret_cast<const uint64_t *>(kh + r * D + ic);
                const uint64_t q2 = *reinterpret_cast<const uint64_t *>(qh + r * D + ic);
                uint64_t xk2 = 0, xq2 = 0, xm2 = 0, eq2;
                if (!slow) {
                    float t0, t1;
                    upk2(mul2(add2(g2, ngm2), l2e2), t0, t1);  // (G - G_mid) log2(e)
                    const uint64_t ep2 = pk2(ex2_approx(t0), ex2_approx(t1));
                    const uint64_t em2 = pk2(ex2_approx(-t0), ex2_approx(-t1));
                    xk2 = mul2(k2, ep2);
                    xq2 = mul2(q2, ep2);
                    xm2 = mul2(k2, em2);
                    eq2 = mul2(ep2, eg2);
                } else {
                    float g0, g1;
                    upk2(g2, g0, g1);
                    eq2 = pk2(__expf(g0), __expf(g1));
                }
                float xp0, xp1;
                upk2(mul2(mul2(sc2, q2), eq2), xp0, xp1);
                *reinterpret_cast<uint32_t *>(blk + WS_QP + umma::sw128_offset<2>(CH, r, ic)) = umma::pack_bf16(xp0, xp1);
                upk2(xk2, xk[j][0], xk[j][1]);
                upk2(xq2, xq[j][0], xq[j][1]);
                upk2(xm2, xm[j][0], xm[j][1]);
                if (!slow) {  // fp32 K+ and K- for P5, over the k^ and G they were formed from
                    *reinterpret_cast<uint64_t *>(kh + r * D + ic) = xk2;
                    *reinterpret_cast<uint64_t *>(G + r * D + ic) = xm2;
                }
            }
        };
        auto store = [&]() {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int r = warp + 16 * j;
                *reinterpret_cast<uint2 *>(X1 + umma::sw128_offset<4>(128, r, c2)) =
                    make_uint2(umma::to_tf32(xk[j][0]), umma::to_tf32(xk[j][1]));
                *reinterpret_cast<uint2 *>(X1 + umma::sw128_offset<4>(128, CH + r, c2)) =
                    make_uint2(umma::to_tf32(xq[j][0]), umma::to_tf32(xq[j][1]));
                *reinterpret_cast<uint2 *>(Km + umma::sw128_offset<4>(CH, r, c2)) =
                    make_uint2(umma::to_tf32(xm[j][0]), umma::to_tf32(xm[j][1]));
            }
        };
        auto mma = [&](int hh) {  // [A; Qk] (+)= [K+; Q+] K-^T over the 64 channels of half hh
            fence_proxy_async_smem();
            umma::fence_before();
            __syncthreads();
            umma::fence_after();
            if (tid == 0) {
                const uint32_t id = umma::idesc(umma::kTF32, 128, CH);
                const uint64_t dX = umma::sdesc_k(X1, 128, 0), dM = umma::sdesc_k(Km, CH, 0);
#pragma unroll
                for (int ks = 0; ks < 64 / 8; ++ks)
                    umma::mma_tf32(tmem, umma::sdesc_at(dX, 128, ks), umma::sdesc_at(dM, CH, ks), id, hh > 0 || ks > 0);
                umma::commit(bar);
            }
        };
        form(0);
        if (!slow) {
            store();
            mma(0);
            form(1);
            ok = wait_all(bar, phase);  // the half-0 MMAs have read the tiles
            phase ^= 1;
            umma::fence_after();
            if (ok) {
                store();
                mma(1);
                ok = wait_all(bar, phase);
                phase ^= 1;
                umma::fence_after();
            }
        } else {
            form(1);
            __syncthreads();
        }
    }
    // ---- P3: A (strict lower, fp32 in smem) and Qk (scaled, lower with the fp32 diagonal, tf32 tile) ----
    // A [64][AST] and Inv [64][IST] (lower block triangle): on the fast path A goes over q^ (dead) and Inv over
    // the [K+; Q+] tile, so that A is written while other warps may still read that tile; the wide-decay path
    // still reads q^ here and keeps the other order
    float *A = reinterpret_cast<float *>(sm + (slow ? I_A : I_Q));
    float *Inv = reinterpret_cast<float *>(sm + (slow ? I_INV : I_A));
    uint8_t *Qks = sm + I_QKS;  // Qk tile staging (read by the copy-out before the next item rewrites it)
    if (ok && !slow) {
        float v[32];
        const int quad = warp & 3, half = (warp >> 2) & 1;  // warps 0-7: lanes 32*quad.., columns 32*half..
        if (warp < 8) {
            umma::ld32(tmem + ((uint32_t)(32 * quad) << 16) + 32 * half, v);
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
                const float dg = a.scale * qkd[r];
#pragma unroll
                for (int t = 0; t < 32; t += 4) {
                    float x4[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int s_ = 32 * half + t + u;
                        x4[u] = s_ < r ? a.scale * v[t + u] : (s_ == r ? dg : 0.f);
                    }
                    umma::st_tf32x4(Qks, CH, r, 32 * half + t, x4[0], x4[1], x4[2], x4[3]);
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
            umma::st_tf32(Qks, CH, r, s_, s_ <= r ? a.scale * accQ : 0.f);
        }
    }
    fence_proxy_async_smem();  // the Qk staging is read by the async proxy below
    if (__syncthreads_or(!ok)) {
        ok = false;
        break;
    }
    if (tid == 0) {  // Qk tile to the workspace
        bulk_s2g(blk + WS_QK, Qks, CH * CH * 4);
        bulk_commit();
    }
    // ---- P4: T = (I + diag(beta) A)^{-1} diag(beta), blocked by 16 ----
    // L = I + diag(beta) A; Inv = L^{-1}, of which only the lower block triangle is formed (the blocks above
    // the diagonal are zero).  Diagonal 16x16 blocks by substitution, one column per thread.
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
        for (int r = 0; r < 16; ++r) Inv[(base + r) * IST + base + col] = x[r];
    }
    __syncthreads();
    // Off-diagonal blocks (i, j = i - d) by distance d:  P_i = diag(beta_i) sum_{k=j}^{i-1} A_ik Inv_kj, then
    // Inv_ij = -Inv_ii P_i.  Each thread forms one row and four columns of a block; a warp covers 8 rows x 16
    // columns, so the row-stride-68 reads of A and Inv_ii fall in distinct banks.
    float *P = reinterpret_cast<float *>(sm + I_T);  // [3][16][16] temporaries (K- is dead)
#pragma unroll
    for (int d = 1; d < 4; ++d) {
        const int nb = 4 - d;  // blocks (i, i-d) for i = d..3
        const bool act = tid < nb * 64;
        const int bi = tid >> 6, rr = (tid >> 2) & 15, c4 = (tid & 3) * 4;
        const int i = bi + d, j = i - d;
        if (act) {
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int kk = 0; kk < d; ++kk) {
                const int k = j + kk;
#pragma unroll
                for (int t = 0; t < 16; ++t) {
                    const float av = A[(16 * i + rr) * AST + 16 * k + t];
                    const float4 iv = *reinterpret_cast<const float4 *>(Inv + (16 * k + t) * IST + 16 * j + c4);
                    acc.x = fmaf(av, iv.x, acc.x);
                    acc.y = fmaf(av, iv.y, acc.y);
                    acc.z = fmaf(av, iv.z, acc.z);
                    acc.w = fmaf(av, iv.w, acc.w);
                }
            }
            const float br = beta[16 * i + rr];
            *reinterpret_cast<float4 *>(P + bi * 256 + rr * 16 + c4) =
                make_float4(br * acc.x, br * acc.y, br * acc.z, br * acc.w);
        }
        __syncthreads();
        if (act) {
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int t = 0; t < 16; ++t) {
                const float lv = Inv[(16 * i + rr) * IST + 16 * i + t];
                const float4 pv = *reinterpret_cast<const float4 *>(P + bi * 256 + t * 16 + c4);
                acc.x = fmaf(lv, pv.x, acc.x);
                acc.y = fmaf(lv, pv.y, acc.y);
                acc.z = fmaf(lv, pv.z, acc.z);
                acc.w = fmaf(lv, pv.w, acc.w);
            }
            *reinterpret_cast<float4 *>(Inv + (16 * i + rr) * IST + 16 * j + c4) =
                make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
        }
        __syncthreads();
    }
    uint8_t *Tt = sm + I_T;  // T tf32 [64 r][64 s]: the B operand of W^T = K+^T T^T (K-major: row r, K = s)
    for (int idx = tid; idx < CH * 16; idx += NTI) {
        const int r = idx >> 4, s0 = (idx & 15) * 4;
        const float4 iv = (s0 >> 4) > (r >> 4) ? make_float4(0.f, 0.f, 0.f, 0.f)
                                               : *reinterpret_cast<const float4 *>(Inv + r * IST + s0);
        umma::st_tf32x4(Tt, CH, r, s0, iv.x * beta[s0], iv.y * beta[s0 + 1], iv.z * beta[s0 + 2], iv.w * beta[s0 + 3]);
    }
    __syncthreads();  // A / Inv are dead: Ktil^T may be staged over them
    // ---- P5: (k exp G)^T tile (A operand) and the Ktil^T workspace tile, 4 tokens per item ----
    uint8_t *Kpt = sm + I_Q;
    uint8_t *Kts = sm + I_A;
    for (int idx = tid; idx < D * 16; idx += NTI) {
        const int i = idx & 127, r0 = (idx >> 7) * 4;
        float kp[4], kt[4];
        if (!slow) {  // k exp(G) = K+ exp(G_mid), k exp(G_last - G) = K- exp(G_last - G_mid)
            const float em = eGm[i], el = eglm[i];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                kp[u] = kh[(r0 + u) * D + i] * em;
                kt[u] = G[(r0 + u) * D + i] * el;
            }
        } else {
            const float glast = G[(CH - 1) * D + i];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float g = G[(r0 + u) * D + i], k_ = kh[(r0 + u) * D + i];
                kp[u] = k_ * __expf(g);
                kt[u] = k_ * __expf(glast - g);
            }
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
        const uint64_t dT = umma::sdesc_k(Tt, CH, 0), dKp = umma::sdesc_k(Kpt, D, 0), dV = umma::sdesc_k(Vt, D, 0);
#pragma unroll
        for (int ks = 0; ks < CH / 8; ++ks) {
            const uint64_t bt = umma::sdesc_at(dT, CH, ks);
            umma::mma_tf32(tmem + 64, umma::sdesc_at(dKp, D, ks), bt, id, ks > 0);
            umma::mma_tf32(tmem + 128, umma::sdesc_at(dV, D, ks), bt, id, ks > 0);
        }
        umma::commit(bar);
    }
    if (tid == 0) {  // Ktil^T tile to the workspace (its staging is not reused)
        bulk_s2g(blk + WS_KT, Kts, D * CH * 4);
        bulk_commit();
    }
    if (tid == NTI - 1 && has_next) load_meta(next, &meta[(it + 1) & 1]);  // while every warp waits for the MMAs
    ok = wait_all(bar, phase);
    phase ^= 1;
    umma::fence_after();
    if (!ok) break;
    // ---- P6: -W (bf16 tile [64 r][128 i]) and U' (fp32 [64 r][128 j]) via smem staging ----
    uint8_t *Wst = sm + I_K;
    float *Ust = reinterpret_cast<float *>(sm + I_VT);  // the V^T tile is dead once the P5 MMAs are done
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
    // The next item's loads start here: its rows go to the raw region (every MMA is done and, once the
    // Ktil^T and Qk copies have been read, nothing else lives there) and its decay logits to the G region
    // (dead after P5).  The -W and U' copy-outs are waited for at the start of the next item.  Its beta logit
    // is fetched into a register meanwhile.
    const ItemMeta mn = meta[(it + 1) & 1];
    const int hn = next % H;
    if (tid == 0) {
        if (has_next) {
            bulk_wait_read_all();  // the Ktil^T and Qk copies
            issue_rows(mn, hn);
            issue_logits(mn, hn);
            in_flight = true;
        }
        bulk_s2g(blk + WS_W, Wst, CH * D * 2);  // -W and U' to the workspace
        bulk_s2g(blk + WS_UP, Ust, CH * D * 4);
        bulk_commit();
    }
    if (has_next) {
        blogit = (tid < CH && tid < mn.n) ? a.b[(size_t)(mn.t0 + tid) * H + hn] : (uint16_t)0;
    }

    // raw conv windows at a checkpoint boundary / at the sequence end (as the SIMT path); the item's
    // metadata is read again here rather than kept in registers across the item
    {
        const ItemMeta me = meta[it & 1];
        const int32_t flag = wsp<int32_t>(a, L.off_flags)[me.seq];
        const int64_t pend = me.p0 + me.n;
        int wslot[2] = {-1, -1};
        if (a.interval > 0 && pend % a.interval == 0 && !(flag & kSeqCkptBad)) {
            const int64_t jj = pend / a.interval - me.start / a.interval - 1;
            const int s_ = a.ckpt_slots[a.ckpt_offsets[me.seq] + jj];
            if (s_ >= a.num_slots || s_ < -1) {
                if (tid == 0) set_status(a.status, KDA_DEV_BAD_SLOT);
            } else {
                wslot[0] = s_;
            }
        }
        if (pend == me.start + me.len) wslot[1] = a.dst[me.seq];
        const int hh = item - (item / H) * H;
        for (int wi = 0; wi < 2; ++wi) {
            if (wslot[wi] < 0) continue;
            uint4 *cw = reinterpret_cast<uint4 *>(a.conv + ((size_t)wslot[wi] * H + hh) * (kConvW - 1) * CC);
            if (tid < 3 * CC / 8) cw[tid] = wstash[tid];
        }
    }
    // (no barrier: the window stash and this item's metadata are rewritten only after the next item's first
    // barrier, and thread 0 waits there for the copy-outs that read this item's staging)
    }  // item loop
    if (tid == 0) bulk_wait_all();  // the last item's copy-outs read this CTA's shared memory
    if (!ok && tid == 0) {
        set_status(a.status, KDA_DEV_TIMEOUT);
        bulk_wait_all();                          // copies that still read this CTA's shared memory
        if (in_flight) mbar_wait(bar_in, ph_in);  // loads issued for an item that never ran (bounded)
    }
    __syncthreads();
    if (warp == 0) umma::dealloc(tmem, 256);
}

}  // namespace tc

namespace tc {

// State kernel smem (bytes, from a 1024-aligned base)
constexpr uint32_t S_ST = 0;          // S^T bf16 tile [128 j][128 i]: A operand of U^T = S^T (-W)^T, O^T = S^T Q+^T
constexpr uint32_t S_OPS = 32768;     // one chunk's workspace block (Qk, -W, Q+, Ktil^T, gl, U'), WS_BLOCK bytes
constexpr uint32_t S_UT32 = 148480;   // U^T tf32 tile [128 j][64 r]: A operand of S^T += U^T Ktil, O^T += U^T Qk^T
constexpr uint32_t S_OST = 181248;    // O staging fp32 [32 r][OST] of the output warps, half a chunk at a time
constexpr int OST = 132;              // (row stride 132: conflict-free)
constexpr uint32_t S_QP2 = 198656;    // the second Q+ buffer (the first is in the chunk block): bf16 [64 r][128 i]
constexpr uint32_t S_NW = 215040;     // RMSNorm weight [128]
constexpr uint32_t S_GLN = 215552;    // exp(G_last) of chunk c [2][128], by chunk parity
constexpr uint32_t S_MISC = 216576;   // barriers, tensor-memory address
constexpr uint32_t S_SMEM = S_MISC + 256 + 1024;
static_assert(S_OPS + WS_BLOCK <= S_UT32 && S_UT32 % 1024 == 0, "state smem layout");
static_assert(S_UT32 + D * CH * 4 <= S_OST && S_OST + 32 * OST * 4 <= S_QP2, "state smem layout");
static_assert(S_QP2 % 1024 == 0 && S_QP2 + CH * D * 2 <= S_NW, "state smem layout");
static_assert(S_NW + D * 4 <= S_GLN && S_GLN + 2 * D * 4 <= S_MISC, "state smem layout");
constexpr int NCW = 8;                // chain warps: two per tensor-memory lane quadrant
constexpr int NOW = 8;                // output warps: two per lane quadrant
constexpr int NTS = 32 * (NCW + NOW);
static_assert(NCW * 32 == 256 && NOW * 32 == 256, "the named barriers below count 256 threads each");

// TMEM columns: S^T [0,128), U^T [128,192), O^T in two buffers [192,256) and [256,320)
constexpr uint32_t T_S = 0, T_U = 128, T_O = 192, T_COLS = 512;

// Barrier 1 over the 256 chain threads, barrier 2 over the 256 output threads (each group runs its own loop).
__device__ __forceinline__ void state_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
__device__ __forceinline__ bool state_sync_or(bool p) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred pi, po;\n setp.ne.u32 pi, %1, 0;\n bar.red.or.pred po, 1, 256, pi;\n selp.u32 %0, 1, 0, po;\n}"
        : "=r"(r)
        : "r"((uint32_t)p)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ bool out_sync_or(bool p) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred pi, po;\n setp.ne.u32 pi, %1, 0;\n bar.red.or.pred po, 2, 256, pi;\n selp.u32 %0, 1, 0, po;\n}"
        : "=r"(r)
        : "r"((uint32_t)p)
        : "memory");
    return r != 0;
}

// The sequential chunk pass of one (sequence, head).  The chain warps run the recurrence with S^T in tensor
// memory, kept decayed by the NEXT chunk's exp(G_last) so that the chunk update is one accumulating MMA:
//   U^T  = S^T (-W)^T                 (MMA, no accumulate)
//   U    = U' + U^T read back         -> tf32 operand tile
//   S^T += U^T Ktil                   (MMA; S^T already holds S^T diag(exp(G_last)))
//   S pass: the bf16 operand tile of the new S, which the next chunk's first MMAs read; then, once those are
//   issued and while they run, the checkpoint and S^T diag(exp(G_last of the next chunk)) back to tensor
//   memory (or the final state to dst).
// The output MMAs O^T = S^T Q+^T + U^T Qk^T go to one of two tensor-memory buffers, which the eight output warps
// read themselves, half a chunk at a time: they apply the gated RMSNorm and store y while the chain goes on, and
// release the buffer for the chunk after next.  Each chain warp owns one lane quadrant (32 value channels) and
// half of the columns: 64 key channels of S, 32 tokens of U.  The chunk block arrives in bulk copies, each
// issued as soon as the chunk before no longer reads its region; Q+ has two buffers and is copied two chunks
// ahead, so that the first O^T MMAs follow the U^T ones at once.
__global__ void __launch_bounds__(NTS, 1) prefill_state_tc_kernel(const PrefillArgs a, const Layout2 L) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int H = a.H, CC = 3 * D;
    const int n = blockIdx.x, h = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int32_t flag = wsp<int32_t>(a, L.off_flags)[n];
    if (flag & kSeqInvalid) return;
    const int src = a.src[n], dst = a.dst[n];  // validated by the table kernel
    uint8_t *Sst = sm + S_ST;
    uint8_t *ops = sm + S_OPS;
    uint8_t *Ut32 = sm + S_UT32;
    float *Ost = reinterpret_cast<float *>(sm + S_OST);
    float *nw = reinterpret_cast<float *>(sm + S_NW);
    float *gln = reinterpret_cast<float *>(sm + S_GLN);
    uint64_t *bar_w = reinterpret_cast<uint64_t *>(sm + S_MISC);  // -W of a chunk
    uint64_t *bar_u = bar_w + 1;                                    // U'
    uint64_t *bar_b = bar_w + 2;                                    // Qk and Ktil^T (+ exp(G_last))
    uint64_t *bar_mma = bar_w + 3;                                  // the U^T and the S^T MMAs
    uint64_t *bar_o = bar_w + 4;      // [2] the O^T MMAs of a chunk into buffer b
    uint64_t *bar_ofree = bar_w + 6;  // [2] buffer b read by the output warps (one arrival per output warp)
    uint64_t *bar_q = bar_w + 8;      // [2] Q+ of a chunk in buffer b (chunk c of this launch: b = (c - cb) & 1)
    uint32_t *tmem_s = reinterpret_cast<uint32_t *>(sm + S_MISC + 128);
    auto qpbuf = [&](int b) { return b ? sm + S_QP2 : ops + WS_QP; };
    const int64_t start = a.start_pos[n];
    const int32_t c0 = wsp<int32_t>(a, L.off_seqc)[n], c1 = wsp<int32_t>(a, L.off_seqc)[n + 1];
    // this launch's chunks of the sequence: [cb, ce) = [c0, c1) within [seg_lo, seg_hi).  The state enters
    // from the source slot at the sequence's first chunk, else from the carry written by the launch before;
    // it leaves to the destination slot at the last chunk, else to the carry.  An empty sequence passes its
    // state and window through in the launch of the first segment.
    const bool empty = c0 == c1;
    const int32_t cb = max(c0, a.seg_lo), ce = min(c1, a.seg_hi);
    if (empty ? a.seg_lo != 0 : cb >= ce) return;
    const bool first = cb == c0, last = ce == c1;
    float *carry = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(a.ws) + L.off_carry) + ((size_t)n * H + h) * D * D;
    const ChunkEnt *ent = wsp<ChunkEnt>(a, L.off_ent);
    const int64_t *pos = wsp<int64_t>(a, L.off_pos);
    const uint8_t *blk0 = reinterpret_cast<const uint8_t *>(a.ws) + L.off_blk;
    auto blk_of = [&](int32_t c) { return blk0 + ((size_t)c * H + h) * WS_BLOCK; };
    // -W is copied as soon as the U^T MMAs are done with it.  Q+ has two buffers, so that the Q+ of chunk
    // c + 2 is copied once the S^T commit of chunk c (which covers the O^T MMAs that read its buffer) is seen:
    // it is in place when its chunk starts
    auto issue_w = [&](int32_t c) {
        mbar_arrive_expect_tx(bar_w, CH * D * 2);
        bulk_g2s(ops + WS_W, blk_of(c) + WS_W, CH * D * 2, bar_w);
    };
    auto issue_qp = [&](int32_t c) {
        const int b = (c - cb) & 1;
        mbar_arrive_expect_tx(bar_q + b, CH * D * 2);
        bulk_g2s(qpbuf(b), blk_of(c) + WS_QP, CH * D * 2, bar_q + b);
    };
    auto issue_u = [&](int32_t c) {
        mbar_arrive_expect_tx(bar_u, CH * D * 4);
        bulk_g2s(ops + WS_UP, blk_of(c) + WS_UP, CH * D * 4, bar_u);
    };
    auto issue_b = [&](int32_t c) {
        mbar_arrive_expect_tx(bar_b, CH * CH * 4 + D * CH * 4 + D * 4);
        bulk_g2s(ops + WS_QK, blk_of(c) + WS_QK, CH * CH * 4, bar_b);
        bulk_g2s(ops + WS_KT, blk_of(c) + WS_KT, D * CH * 4 + D * 4, bar_b);  // Ktil^T and exp(G_last)
    };

    // thread 0's record of the copies it issued and has not yet seen complete, with the parity of the phase
    // that completes each (read only on the exit after a timed-out wait)
    bool out_w = false, out_u = false, out_b = false;
    uint32_t par_w = 0, par_u = 0, par_b = 0;
    uint32_t out_q = 0, par_q = 0;  // bit b: a Q+ copy into buffer b in flight / the parity of its phase
    if (warp == 0) umma::alloc(tmem_s, T_COLS);
    for (int jj = tid; jj < D; jj += NTS) nw[jj] = __ldg(a.norm_w + jj);
    if (tid == 0) {
        for (int b = 0; b < 4; ++b) mbar_init(bar_w + b, 1);
        mbar_init(bar_q, 1);
        mbar_init(bar_q + 1, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar_o + b, 1);
            mbar_init(bar_ofree + b, NOW);
        }
        fence_mbar_init();
        if (!empty) {
            issue_w(cb);
            issue_qp(cb);
            issue_u(cb);
            issue_b(cb);
            out_w = out_u = out_b = true;
            out_q = 1u;
            if (cb + 1 < ce) {
                issue_qp(cb + 1);
                out_q = 3u;
            }
        }
    }
    umma::fence_before();
    __syncthreads();
    umma::fence_after();
    const uint32_t tmem = *tmem_s;

    if (warp < NCW) {
        // ================================ chain warps ================================
        const int quad = warp & 3, part = warp >> 2;
        const int j = 32 * quad + lane;  // this thread's value channel = tensor-memory lane
        const uint32_t lane_off = (uint32_t)(32 * quad) << 16;
        const int i0 = 64 * part;        // this thread's key channels of S: i0 .. i0 + 63
        const int r0 = 32 * part;        // this thread's tokens of U: r0 .. r0 + 31
        // initial state: its bf16 operand tile, and S^T diag(exp(G_last of the first chunk)) in tensor memory
        {
            const float *gl0 = !empty ? reinterpret_cast<const float *>(blk_of(cb) + WS_GL) : nullptr;
            float v[32];
            for (int g = 0; g < 2; ++g) {
                const int ig = i0 + 32 * g;
                if (first) {
#pragma unroll
                    for (int t = 0; t < 32; ++t)
                        v[t] = src >= 0 ? load_state(a.S, a.state_bf16, (((size_t)src * H + h) * D + ig + t) * D + j)
                                        : 0.f;
                } else {
#pragma unroll
                    for (int t = 0; t < 32; ++t) v[t] = carry[(size_t)(ig + t) * D + j];
                }
                if (empty) {  // empty sequence: the state passes through unchanged
#pragma unroll
                    for (int t = 0; t < 32; ++t)
                        store_state(a.S, a.state_bf16, (((size_t)dst * H + h) * D + ig + t) * D + j, v[t]);
                    continue;
                }
#pragma unroll
                for (int t = 0; t < 32; t += 8) umma::st_bf16x8(Sst, D, j, ig + t, v + t);
#pragma unroll
                for (int t = 0; t < 32; ++t) v[t] *= __ldg(gl0 + ig + t);
                umma::st32(tmem + lane_off + T_S + ig, v);
            }
            if (empty) {  // and so does the window
                uint16_t *cw = a.conv + ((size_t)dst * H + h) * (kConvW - 1) * CC;
                for (int idx = tid; idx < (kConvW - 1) * CC; idx += 32 * NCW)
                    cw[idx] = src >= 0 ? a.conv[((size_t)src * H + h) * (kConvW - 1) * CC + idx] : (uint16_t)0;
            }
        }
        fence_proxy_async_smem();
        umma::fence_before();
        state_sync();
        umma::fence_after();
        uint32_t ph_w = 0, ph_u = 0, ph_b = 0, ph_m = 0;
        bool ok = true, t0ok = true;  // t0ok: thread 0's waits on the output warps' buffer releases
        // checkpoint boundaries: a running next boundary, its slot fetched one boundary ahead (no division in
        // the loop); chunk entries are fetched one chunk ahead
        // (the boundaries at or before this launch's first position belong to the chunks before it)
        const bool want_ck = a.interval > 0 && !(flag & kSeqCkptBad) && !empty;
        const int64_t send = start + ((int64_t)a.cu_seqlens[n + 1] - a.cu_seqlens[n]);
        const int64_t pb = !empty ? pos[cb] : start;
        int64_t next_b = want_ck ? (pb / a.interval + 1) * a.interval : INT64_MAX;
        const int32_t *cks = want_ck ? a.ckpt_slots + a.ckpt_offsets[n] : nullptr;
        int jck = want_ck ? (int)(pb / a.interval - start / a.interval) : 0;
        int ck_pre = (want_ck && next_b <= send) ? cks[jck] : -1;
        ChunkEnt e_nx = !empty ? ent[cb] : ChunkEnt{};
        int64_t p_nx = pb;
        int ck_prev = -1;  // checkpoint slot of the chunk before's end
        // The state pass of a chunk (key channels i0 .. i0 + 63 of S^T, in tensor memory) after its bf16 tile:
        // the checkpoint, then S^T diag(exp(G_last of the next chunk)) back to tensor memory when a chunk follows
        // in this launch (gl: its exp(G_last)), else the state to the destination slot or to the carry.
        auto s_rest = [&](int ckp, const float *gl) {
#pragma unroll 1
            for (int g = 0; g < 2; ++g) {
                const int ig = i0 + 32 * g;
                uint32_t r[32];
                umma::ld32_issue(tmem + lane_off + T_S + ig, r);
                umma::wait_ld(r);
                float v[32];
#pragma unroll
                for (int t = 0; t < 32; ++t) v[t] = __uint_as_float(r[t]);
                if (ckp >= 0) {
#pragma unroll
                    for (int t = 0; t < 32; ++t)
                        store_state(a.S, a.state_bf16, (((size_t)ckp * H + h) * D + ig + t) * D + j, v[t]);
                }
                if (gl) {
#pragma unroll
                    for (int t = 0; t < 32; t += 4) {
                        const float4 g4 = *reinterpret_cast<const float4 *>(gl + ig + t);
                        v[t] *= g4.x;
                        v[t + 1] *= g4.y;
                        v[t + 2] *= g4.z;
                        v[t + 3] *= g4.w;
                    }
                    umma::st32_issue(tmem + lane_off + T_S + ig, v);
                } else if (last) {
#pragma unroll
                    for (int t = 0; t < 32; ++t)
                        store_state(a.S, a.state_bf16, (((size_t)dst * H + h) * D + ig + t) * D + j, v[t]);
                } else {
#pragma unroll
                    for (int t = 0; t < 32; ++t) carry[(size_t)(ig + t) * D + j] = v[t];
                }
            }
            umma::wait_st();
        };
        for (int32_t c = cb; c < ce; ++c) {
            const ChunkEnt e = e_nx;
            const int ob = (c - cb) & 1;                        // O^T buffer of this chunk
            const uint32_t opar = (uint32_t)((c - cb) >> 1) & 1u;  // parity of this use of it
            const int64_t pend = p_nx + e.n;
            const bool has_next = c + 1 < ce;
            if (has_next) {
                e_nx = ent[c + 1];
                p_nx = pos[c + 1];
            }
            int ck = -1;  // checkpoint slot of this chunk's end
            if (pend == next_b) {
                if (ck_pre >= 0 && ck_pre < a.num_slots) ck = ck_pre;
                ++jck;
                next_b += a.interval;
                ck_pre = next_b <= send ? cks[jck] : -1;
            }
            const float gnext = (tid < D && has_next) ? __ldg(reinterpret_cast<const float *>(blk_of(c + 1) + WS_GL) + tid)
                                                      : 1.f;
            // ---- U^T = S^T (-W)^T.  If -W never arrives, nothing is committed and every thread's bounded wait
            //      on bar_mma gives up ----
            // ---- U^T = S^T (-W)^T; then, once Q+ is in (copied two chunks ahead) and the output warps have read
            //      this O^T buffer (two chunks ago), O^T = S^T Q+^T (the S^T commit below covers it).  If -W or Q+
            //      never arrives, nothing more is committed and every thread's bounded wait on bar_mma gives up ----
            const uint32_t idp = umma::idesc(umma::kBF16, 128, CH);
            const uint64_t dS = umma::sdesc_k(Sst, D, 0);
            if (tid == 0 && mbar_wait(bar_w, ph_w)) {
                out_w = false;
                const uint64_t dW = umma::sdesc_k(ops + WS_W, CH, 0);
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks)
                    umma::mma_bf16(tmem + T_U, umma::sdesc_at(dS, D, ks), umma::sdesc_at(dW, CH, ks), idp, ks > 0);
                umma::commit(bar_mma);
                const int qb = ob;  // (the same chunk parity)
                const bool okq = mbar_wait(bar_q + qb, opar);
                if (okq) out_q &= ~(1u << qb);
                if (!okq || (c - cb >= 2 && !mbar_wait(bar_ofree + ob, opar ^ 1u))) t0ok = false;
                umma::fence_after();
                if (t0ok) {
                    const uint32_t tob = tmem + T_O + 64u * (uint32_t)ob;
                    const uint64_t dQ = umma::sdesc_k(qpbuf(qb), CH, 0);
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks)
                        umma::mma_bf16(tob, umma::sdesc_at(dS, D, ks), umma::sdesc_at(dQ, CH, ks), idp, ks > 0);
                }
            }
            ph_w ^= 1;
            // the rest of the state pass of the chunk before, while the MMAs above run: its checkpoint, and
            // S^T diag(exp(G_last of this chunk)) back to tensor memory for this chunk's S^T MMA
            if (c > cb) s_rest(ck_prev, gln + (c & 1) * D);
            // each thread waits for U^T itself; a timed-out wait is voted on at the barrier after the U tiles
            ok = mbar_wait(bar_mma, ph_m);
            ph_m ^= 1;
            umma::fence_after();
            if (tid == 0 && ok && has_next) {  // the U^T MMAs no longer read -W
                issue_w(c + 1);
                out_w = true;
                par_w = ph_w;
            }
            // ---- U = U' + U^T -> its tf32 operand tile (this thread: tokens r0 .. r0 + 31) ----
            const bool oku = mbar_wait(bar_u, ph_u);
            if (oku) out_u = false;
            ok = __all_sync(0xffffffffu, oku && ok);  // warp-uniform: the load is a warp operation
            ph_u ^= 1;
            if (ok) {
                const float *up = reinterpret_cast<const float *>(ops + WS_UP);
                float v[32];
#pragma unroll
                for (int t = 0; t < 32; ++t) v[t] = up[(r0 + t) * D + j];  // in flight with the U^T load
                uint32_t r[32];
                umma::ld32_issue(tmem + lane_off + T_U + r0, r);
                umma::wait_ld(r);
#pragma unroll
                for (int t = 0; t < 32; ++t) v[t] += __uint_as_float(r[t]);
#pragma unroll
                for (int t = 0; t < 32; t += 4)
                    umma::st_tf32x4(Ut32, D, j, r0 + t, v[t], v[t + 1], v[t + 2], v[t + 3]);
            }
            if (tid < D) gln[((c + 1) & 1) * D + tid] = gnext;

            fence_proxy_async_smem();
            umma::fence_before();
            ok = !state_sync_or(!(ok && t0ok));
            umma::fence_after();
            if (!ok) break;
            // ---- S^T += U^T Ktil, then O^T += U^T Qk^T ----
            if (tid == 0) {
                if (has_next) {  // U' has been read by every thread
                    issue_u(c + 1);
                    out_u = true;
                    par_u = ph_u;
                }
                const bool okb = mbar_wait(bar_b, ph_b);
                if (okb) {
                    out_b = false;
                    const uint32_t ids = umma::idesc(umma::kTF32, 128, D);
                    const uint64_t dU = umma::sdesc_k(Ut32, D, 0), dK = umma::sdesc_k(ops + WS_KT, D, 0);
#pragma unroll
                    for (int ks = 0; ks < CH / 8; ++ks)
                        umma::mma_tf32(tmem + T_S, umma::sdesc_at(dU, D, ks), umma::sdesc_at(dK, D, ks), ids, true);
                    umma::commit(bar_mma);  // the S pass needs only S^T
                    const uint32_t ido = umma::idesc(umma::kTF32, 128, CH);
                    const uint32_t tob = tmem + T_O + 64u * (uint32_t)ob;
                    const uint64_t dQk = umma::sdesc_k(ops + WS_QK, CH, 0);
#pragma unroll
                    for (int ks = 0; ks < CH / 8; ++ks)
                        umma::mma_tf32(tob, umma::sdesc_at(dU, D, ks), umma::sdesc_at(dQk, CH, ks), ido, true);
                    umma::commit(bar_o + ob);  // covers both rounds of O^T MMAs: the output warps take it from here
                }
            }
            ph_b ^= 1;
            // each thread waits for S^T itself; the vote is taken at the end of the chunk
            ok = __all_sync(0xffffffffu, mbar_wait(bar_mma, ph_m));
            ph_m ^= 1;
            umma::fence_after();
            if (tid == 0 && ok && c + 2 < ce) {  // every MMA before the S^T commit is done: this Q+ buffer is free
                issue_qp(c + 2);
                out_q |= 1u << ob;
                par_q = (par_q & ~(1u << ob)) | ((opar ^ 1u) << ob);
            }

            // ---- S pass, the part the next chunk's first MMAs wait for (this thread: key channels i0 .. i0 + 63):
            //      the bf16 operand tile of the new state.  The rest (checkpoint, decay, final store) follows the
            //      barrier below, or the next chunk's MMA issue. ----
            if (ok && has_next) {
#pragma unroll 1
                for (int g = 0; g < 2; ++g) {
                    uint32_t r[32];
                    umma::ld32_issue(tmem + lane_off + T_S + i0 + 32 * g, r);
                    umma::wait_ld(r);
                    float v[32];
#pragma unroll
                    for (int t = 0; t < 32; ++t) v[t] = __uint_as_float(r[t]);
#pragma unroll
                    for (int t = 0; t < 32; t += 8) umma::st_bf16x8(Sst, D, j, i0 + 32 * g + t, v + t);
                }
            }
            // Qk and Ktil^T of the next chunk, once the O^T MMAs that read Qk are done (thread 0; the S^T MMAs
            // that read Ktil^T are)
            if (tid == 0 && ok && has_next) {
                if (mbar_wait(bar_o + ob, opar)) {
                    issue_b(c + 1);
                    out_b = true;
                    par_b = ph_b;
                } else {
                    t0ok = false;
                }
            }
            fence_proxy_async_smem();
            umma::fence_before();
            ok = !state_sync_or(!(ok && t0ok));
            umma::fence_after();
            if (!ok) break;
            ck_prev = ck;
        }
        if (ok && ce > cb) s_rest(ck_prev, nullptr);  // the last chunk's checkpoint and the final (or carried) state
        if (!ok && tid == 0) {
            set_status(a.status, KDA_DEV_TIMEOUT);
            // copies still in flight into this CTA's shared memory land before it exits (short bounded waits)
            constexpr uint64_t kDrainNs = 10000000ull;
            if (out_w) mbar_wait(bar_w, par_w, kDrainNs);
            for (int b = 0; b < 2; ++b)
                if (out_q >> b & 1u) mbar_wait(bar_q + b, par_q >> b & 1u, kDrainNs);
            if (out_u) mbar_wait(bar_u, par_u, kDrainNs);
            if (out_b) mbar_wait(bar_b, par_b, kDrainNs);
        }
    } else {
        // ================================ output warps ================================
        // The O^T buffer is staged and normalised in two halves of 32 tokens.  Staging: warp ow takes lane
        // quadrant ow % 4 (NCW % 4 == 0) and 16 tokens (ow / 4) of the half; the gated RMSNorm: tokens ow,
        // ow + 8, ..., one warp per token
        const int ow = warp - NCW, oq = ow & 3, oh = ow >> 2;
        uint2 zr[8];
        auto fetch_gates = [&](const ChunkEnt &e) {  // the output gate of this warp's tokens of a chunk
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int r = ow + 8 * k;
                zr[k] = (a.z && r < e.n)
                            ? __ldg(reinterpret_cast<const uint2 *>(a.z + ((size_t)(e.t0 + r) * H + h) * D) + lane)
                            : make_uint2(0u, 0u);
            }
        };
        ChunkEnt e_nx = !empty ? ent[cb] : ChunkEnt{};
        for (int32_t c = cb; c < ce; ++c) {
            const ChunkEnt e = e_nx;
            if (c + 1 < ce) e_nx = ent[c + 1];  // in flight while this chunk is processed
            fetch_gates(e);  // in flight while the O^T of this chunk is awaited and staged
            const int ob = (c - cb) & 1;
            const uint32_t opar = (uint32_t)((c - cb) >> 1) & 1u;
            // O^T of this chunk from its tensor-memory buffer (this warp: value channels 32 oq .. 32 oq + 31,
            // tokens 32 oh .. 32 oh + 31)
            const bool okw = __all_sync(0xffffffffu, mbar_wait(bar_o + ob, opar));
            if (out_sync_or(!okw)) {  // every output warp before the staging is rewritten; a timeout ends them all
                if (tid == 32 * NCW) set_status(a.status, KDA_DEV_TIMEOUT);
                break;
            }
            umma::fence_after();
            const float4 w4 = *reinterpret_cast<const float4 *>(nw + 4 * lane);
#pragma unroll
            for (int p = 0; p < 2; ++p) {
                {   // tokens 32 p + 16 oh .. 32 p + 16 oh + 15 of value channels 32 oq .. 32 oq + 31
                    uint32_t va[16];
                    umma::ld16_issue(tmem + ((uint32_t)(32 * oq) << 16) + T_O + 64u * (uint32_t)ob + 32u * (uint32_t)p +
                                         16u * (uint32_t)oh,
                                     va);
                    umma::wait_ld16(va);
                    const int jo = 32 * oq + lane;
#pragma unroll
                    for (int t = 0; t < 16; ++t) Ost[(16 * oh + t) * OST + jo] = __uint_as_float(va[t]);
                }
                if (p == 1) {  // this warp's parts of the buffer are read
                    umma::fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_expect_tx(bar_ofree + ob, 0);
                }
                out_sync_or(false);  // these 32 tokens are staged
                // the 4 rows are read before any y store (the stores could otherwise be taken to alias the
                // staging), and their reductions are interleaved
                float4 o4r[4];
                float ss[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    o4r[k] = *reinterpret_cast<const float4 *>(Ost + (ow + 8 * k) * OST + 4 * lane);
                    ss[k] = o4r[k].x * o4r[k].x;
                    ss[k] = fmaf(o4r[k].y, o4r[k].y, ss[k]);
                    ss[k] = fmaf(o4r[k].z, o4r[k].z, ss[k]);
                    ss[k] = fmaf(o4r[k].w, o4r[k].w, ss[k]);
                }
                if (p == 0) out_sync_or(false);  // every warp has read this half before the next is staged
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
#pragma unroll
                    for (int k = 0; k < 4; ++k) ss[k] += __shfl_xor_sync(0xffffffffu, ss[k], o);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int r = 32 * p + ow + 8 * k;
                    const float4 o4 = o4r[k];
                    const float rr = rsqrtf(ss[k] * (1.0f / D) + a.rms_eps);
                    if (r < e.n) {
                        float y0 = o4.x * rr * w4.x, y1 = o4.y * rr * w4.y, y2 = o4.z * rr * w4.z, y3 = o4.w * rr * w4.w;
                        if (a.z) {
                            const uint2 zz = zr[4 * p + k];
                            y0 *= sigmoid_gate(bf2f((uint16_t)(zz.x & 0xffff)));
                            y1 *= sigmoid_gate(bf2f((uint16_t)(zz.x >> 16)));
                            y2 *= sigmoid_gate(bf2f((uint16_t)(zz.y & 0xffff)));
                            y3 *= sigmoid_gate(bf2f((uint16_t)(zz.y >> 16)));
                        }
                        *(reinterpret_cast<uint2 *>(a.y + ((size_t)(e.t0 + r) * H + h) * D) + lane) =
                            make_uint2((uint32_t)f2bf(y0) | ((uint32_t)f2bf(y1) << 16),
                                       (uint32_t)f2bf(y2) | ((uint32_t)f2bf(y3) << 16));
                    }
                }
            }
        }
    }
    umma::fence_before();
    __syncthreads();
    if (warp == 0) umma::dealloc(tmem, T_COLS);
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

// Blocks of the table kernel: one for the tables, and enough for the window snapshot (at most two per SM).
static unsigned table_grid(const PrefillArgs &a, const Layout &L) {
    const long long words = (long long)a.nseq * a.H * L.win_u4;
    const long long copy = std::min<long long>((words + kMaxSeqThreads - 1) / kMaxSeqThreads, 2LL * current_device_sms());
    return (unsigned)(1 + copy);
}

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled, looked up once through the runtime (no link against the driver library).
static EncodeTiledFn tensor_map_encoder() {
    static std::atomic<EncodeTiledFn> cached{nullptr};
    EncodeTiledFn f = cached.load(std::memory_order_acquire);
    if (f) return f;
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !p)
        return nullptr;
    f = reinterpret_cast<EncodeTiledFn>(p);
    cached.store(f, std::memory_order_release);
    return f;
}

// A [T][H][128] bf16 token tensor as a 3-D map (channel, head, token) with boxes of 128 channels x 1 head x
// `rows` tokens; out-of-range tokens read as zeros.
static bool token_map(EncodeTiledFn enc, CUtensorMap *m, const void *base, int H, int64_t T, int rows) {
    const cuuint64_t dims[3] = {(cuuint64_t)tc::D, (cuuint64_t)H, (cuuint64_t)T};
    const cuuint64_t strides[2] = {(cuuint64_t)tc::D * 2, (cuuint64_t)H * tc::D * 2};
    const cuuint32_t box[3] = {(cuuint32_t)tc::D, 1u, (cuuint32_t)rows};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Segmented launches.  With few (sequence, head) chains the state kernel leaves most SMs idle while it walks
// a long chunk chain after the intra kernel.  Such a call is cut into segments of kSegChunks chunks: the intra
// kernel of segment s+1 runs on nsm - chains SMs while the state kernel of segment s runs on the other
// `chains`, on a side stream that waits (events only, no device-side waiting) for the intra kernel of its
// segment.  The state crosses a segment boundary in fp32 through the workspace and sees the same arithmetic
// as at a chunk boundary inside one launch, so the results are identical to a single launch.
constexpr int kSegChunks = 128;
constexpr int64_t kSegMinChunks = 4 * kSegChunks;

struct SideStream {
    std::mutex mu;
    cudaStream_t stream = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};

static SideStream *side_stream(int dev) {
    static SideStream side[64];
    if (dev < 0 || dev >= 64) return nullptr;
    return &side[dev];
}

// The dynamic shared-memory limits of the prefill kernels, once per device (the current one).
static int set_prefill_attributes(int dev) {
    static std::atomic<int> done[64];
    if (done[dev].load(std::memory_order_acquire)) return KDA_OK;
    const int max_smem = 227 * 1024;
    if (cudaFuncSetAttribute(tc::prefill_intra_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, tc::I_SMEM) !=
            cudaSuccess ||
        cudaFuncSetAttribute(tc::prefill_state_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, tc::S_SMEM) !=
            cudaSuccess ||
        cudaFuncSetAttribute(prefill_intra_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem) !=
            cudaSuccess ||
        cudaFuncSetAttribute(prefill_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem) !=
            cudaSuccess)
        return launch_result("prefill: cudaFuncSetAttribute");
    done[dev].store(1, std::memory_order_release);
    return KDA_OK;
}

// The side stream and events of segmented launches on this device, created on first use (caller holds mu).
static int ensure_side_stream(SideStream *ss) {
    if (ss->stream) return KDA_OK;
    if (cudaStreamCreateWithFlags(&ss->stream, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&ss->fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&ss->join, cudaEventDisableTiming) != cudaSuccess)
        return launch_result("prefill: side stream creation");
    return KDA_OK;
}

int prefill_prepare() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return launch_result("prefill: cudaGetDevice");
    if (set_prefill_attributes(dev) != KDA_OK) return KDA_ERR_CUDA;
    if (!tensor_map_encoder()) return fail(KDA_ERR_CUDA, "prefill: cuTensorMapEncodeTiled is not available");
    (void)current_device_sms();
    SideStream *ss = side_stream(dev);
    std::lock_guard<std::mutex> lock(ss->mu);
    return ensure_side_stream(ss);
}

static int launch_prefill_tc(const PrefillArgs &a0, cudaStream_t st) {
    PrefillArgs a = a0;
    a.seg_lo = 0;
    a.seg_hi = INT32_MAX;
    const tc::Layout2 L2 = tc::make_layout2(a.H, a.nseq, a.total_tokens);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return launch_result("prefill: cudaGetDevice");
    if (set_prefill_attributes(dev) != KDA_OK) return KDA_ERR_CUDA;
    if (L2.maxc * a.H > 0x7fffffffLL || a.H > 65535) return fail(KDA_ERR_INVALID_ARG, "prefill: grid too large");
    prefill_table_kernel<<<table_grid(a, tc::as_layout(L2)), kMaxSeqThreads, 0, st>>>(a, tc::as_layout(L2));
    CUtensorMap tq, tk, tv, ta;
    if (a.total_tokens > 0) {
        const EncodeTiledFn enc = tensor_map_encoder();
        if (!enc) return fail(KDA_ERR_CUDA, "prefill: cuTensorMapEncodeTiled is not available");
        if (!token_map(enc, &tq, a.q, a.H, a.total_tokens, tc::RAW_ROWS) ||
            !token_map(enc, &tk, a.k, a.H, a.total_tokens, tc::RAW_ROWS) ||
            !token_map(enc, &tv, a.v, a.H, a.total_tokens, tc::RAW_ROWS) ||
            !token_map(enc, &ta, a.a, a.H, a.total_tokens, tc::CH))
            return fail(KDA_ERR_CUDA, "prefill: tensor map encoding failed");
    }
    const int nsm = current_device_sms();
    const long long chains = (long long)a.nseq * a.H;
    const dim3 gs(a.nseq, a.H);
    if (a.total_tokens == 0 || chains * 4 > nsm || L2.maxc < kSegMinChunks) {
        if (a.total_tokens > 0) {
            const long long items = L2.maxc * a.H;  // an upper bound; the kernel reads the real count
            const unsigned gi = (unsigned)std::min<long long>(items, nsm);  // one CTA per SM
            tc::prefill_intra_tc_kernel<<<gi, tc::NTI, tc::I_SMEM, st>>>(a, L2, tq, tk, tv, ta);
        }
        tc::prefill_state_tc_kernel<<<gs, tc::NTS, tc::S_SMEM, st>>>(a, L2);
        return launch_result("prefill (tensor-core path) launch");
    }
    SideStream *ss = side_stream(dev);
    if (!ss) return fail(KDA_ERR_CUDA, "prefill: no side stream for this device");
    std::lock_guard<std::mutex> lock(ss->mu);  // one segmented call at a time per device: the events are shared
    if (ensure_side_stream(ss) != KDA_OK) return KDA_ERR_CUDA;
    const unsigned gi = (unsigned)(nsm - chains);  // the intra CTAs leave one SM to each state CTA
    bool forked = true;
    for (long long lo = 0; lo < L2.maxc && forked; lo += kSegChunks) {
        a.seg_lo = (int32_t)lo;
        a.seg_hi = (int32_t)std::min<long long>(lo + kSegChunks, INT32_MAX);
        tc::prefill_intra_tc_kernel<<<gi, tc::NTI, tc::I_SMEM, st>>>(a, L2, tq, tk, tv, ta);
        forked = cudaEventRecord(ss->fork, st) == cudaSuccess && cudaStreamWaitEvent(ss->stream, ss->fork, 0) == cudaSuccess;
        if (forked) tc::prefill_state_tc_kernel<<<gs, tc::NTS, tc::S_SMEM, ss->stream>>>(a, L2);
    }
    // the caller's stream always waits for the side stream, also after a failed fork
    const bool joined =
        cudaEventRecord(ss->join, ss->stream) == cudaSuccess && cudaStreamWaitEvent(st, ss->join, 0) == cudaSuccess;
    if (!forked || !joined) return launch_result("prefill: segment fork / join");
    return launch_result("prefill (tensor-core path, segmented) launch");
}

int launch_prefill(const PrefillArgs &a, int dk, int dv, cudaStream_t st) {
    if (use_tensor_cores(dk, dv, a.chunk)) return launch_prefill_tc(a, st);
    const Layout L = make_layout(a.H, dk, dv, a.nseq, a.total_tokens, a.chunk);
    const int C = a.chunk;
    const size_t smem_intra = sizeof(float) * (3 * C * dk + C * (dk + dv) + 2 * C * C + C);
    const int DVT = std::min(dv, 32);
    const size_t smem_state = sizeof(float) * (dk * DVT + 3 * C * dk + C * C + 2 * C * DVT + dk);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return launch_result("prefill: cudaGetDevice");
    if (set_prefill_attributes(dev) != KDA_OK) return KDA_ERR_CUDA;
    if (L.maxc > 0x7fffffffLL || a.H > 65535) return fail(KDA_ERR_INVALID_ARG, "prefill: grid too large");
    prefill_table_kernel<<<table_grid(a, L), kMaxSeqThreads, 0, st>>>(a, L);
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
