/*
 * kda.h -- C ABI of the GB300 (sm_103a) Kimi Delta Attention (KDA) serving hot path.
 *
 * KDA is the gated delta rule with channel-wise decay used by Kimi Linear / Kimi K3:
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T ,   o_t = scale * S_t^T q_t
 *
 * Per request and head it keeps a dk x dv fp32 recurrent state S and a short causal-convolution state
 * ("A Preview of Production-Scale Kimi K3 Support on vLLM", section "The Hardest Part: Prefix Caching
 * for KDA": each KDA layer advances a matrix-like recurrent state together with a short convolution
 * state).  One token, for one head, is processed as:
 *   1. causal conv of width W over the raw q | k | v channels (weights [H][2dk+dv][W], tap W-1 on the
 *      current input, tap 0 on the oldest stored one), then SiLU when conv_silu != 0;
 *   2. q^ = q / sqrt(|q|^2 + l2_eps), k^ likewise (v is the conv output as is);
 *   3. alpha = sigmoid(a) per key channel, beta = sigmoid(b) per head (a, b are logits);
 *   4. the update above;  5. o = scale * S^T q^;
 *   6. y = o / sqrt(mean(o^2) + rms_eps) * norm_weight * sigmoid(z)   (gate factor 1 when z is NULL).
 *
 * All entry points are asynchronous on the given stream, allocate nothing, keep no state between
 * calls, and never synchronise the host, so they may be captured in a CUDA graph.  The caller owns
 * every buffer.  All pointers named "device" must be device (or managed) memory of the current device,
 * 16-byte aligned.  bf16 tensors are passed as their uint16 bit patterns.
 *
 * Errors: problems visible on the host return a kda_status before anything is launched.  Problems only
 * visible on the device (an out-of-range slot index, inconsistent sequence or checkpoint tables) OR a bit into *dev_status (a device int32 the caller
 * zeroes and reads after synchronising) and skip the affected work item; kernels never trap.
 */
#ifndef KDA_H
#define KDA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define KDA_API __attribute__((visibility("default")))
#else
#define KDA_API
#endif

/* Same type as cudaStream_t.  NULL is the legacy default stream. */
typedef struct CUstream_st *kda_stream_t;

/* Host-side return codes. */
enum kda_status {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1,       /* NULL pointer, negative count, misaligned pointer, bad interval */
    KDA_ERR_UNSUPPORTED_SHAPE = 2, /* (dk, dv, conv width, chunk) not compiled in */
    KDA_ERR_WORKSPACE = 3,         /* workspace NULL or smaller than kda_prefill_workspace_bytes() */
    KDA_ERR_CUDA = 4               /* a CUDA launch or attribute call failed */
};

/* Device-side status bits, OR-ed into *dev_status. */
#define KDA_DEV_BAD_SLOT 0x1      /* a slot index outside [0, num_slots) (src may also be -1) */
#define KDA_DEV_BAD_SEQLENS 0x2   /* cu_seqlens not non-decreasing from 0 to total_tokens, or start_pos < 0 */
#define KDA_DEV_BAD_CKPT 0x4      /* ckpt_offsets does not give sequence n exactly its boundary count */
#define KDA_DEV_TIMEOUT 0x10      /* a bounded wait on an asynchronous copy gave up */

/*
 * The state-slot pool ("The Hardest Part: Prefix Caching for KDA": the physical state block is
 * decoupled from the prefix-match unit; a slot here is one state snapshot).  Layout, slot-major:
 *   S    [num_slots][H][dk][dv]         state_dtype (fp32, or bf16 bit patterns); row i = key channel,
 *                                       column j = value channel
 *   conv [num_slots][H][W-1][2dk+dv]    bf16, the last W-1 RAW (pre-conv) q|k|v inputs, oldest first
 * Both device, owned by the caller.  With a bf16 pool ("moonshotai/Kimi-K3" recipe:
 * --mamba-ssm-cache-dtype bfloat16) every kernel computes in fp32 and rounds the state to bf16 (nearest
 * even) where it is stored; this halves the state bytes of a decode step.
 */
enum kda_state_dtype { KDA_STATE_FP32 = 0, KDA_STATE_BF16 = 1 };

typedef struct kda_pool {
    int32_t H, dk, dv, conv_w;  /* heads, key dim, value dim, conv width W */
    int32_t state_dtype;        /* enum kda_state_dtype */
    int32_t reserved;           /* 0 */
    int64_t num_slots;
    void *S;
    uint16_t *conv;
} kda_pool;

/* Layer constants. */
typedef struct kda_params {
    const float *conv_weight; /* device [H][2dk+dv][W] fp32 */
    const float *norm_weight; /* device [dv] fp32 (shared by all heads) */
    float l2_eps;             /* q/k normalisation: x / sqrt(|x|^2 + l2_eps) */
    float rms_eps;            /* output RMSNorm epsilon */
    float scale;              /* readout scale */
    int32_t conv_silu;        /* 1: SiLU after the conv; 0: none */
} kda_params;

/*
 * One decode token for each of n requests, all heads, in one launch: conv, gates, state update,
 * readout and gated RMSNorm fused ("A Preview of Production-Scale Kimi K3 Support on vLLM", section
 * "KDA prefill and decode"; "vLLM Kimi K3 Support", section "Fused Kernels and Metadata Optimization":
 * one launch, no intermediate tensors, no repeated state traffic).
 *   q, k      device [n][H][dk] bf16        v, z  device [n][H][dv] bf16 (z may be NULL: no gate)
 *   a         device [n][H][dk] bf16 (decay logits)   b  device [n][H] bf16 (beta logits)
 *   y         device [n][H][dv] bf16 output
 *   src_slot  device [n] int32: state read from this slot; -1 = fresh request (zero state and window)
 *   dst_slot  device [n] int32: updated state and window written here (src == dst: in place)
 *   dev_status device int32, OR-ed with KDA_DEV_* bits.
 * Within one call no dst slot may repeat and no slot may be the src of one request and the dst of
 * another ("The Hardest Part: Prefix Caching for KDA": same-step reuse is deferred until the copy is
 * safe).  A request with a bad slot index gets y = 0 and no state write.
 * Supported: (dk, dv) in {(16,16), (32,16), (16,32), (64,64), (128,128)}, W = 4.
 */
KDA_API int kda_decode_step(const kda_pool *pool, const kda_params *prm, int32_t n, const uint16_t *q, const uint16_t *k,
                    const uint16_t *v, const uint16_t *a, const uint16_t *b, const uint16_t *z, uint16_t *y,
                    const int32_t *src_slot, const int32_t *dst_slot, int32_t *dev_status, kda_stream_t stream);

/*
 * The input projections of a KDA layer in one GEMM ("A Preview of Production-Scale Kimi K3 Support on
 * vLLM", section "KDA prefill and decode": the input projections and the causal convolution are fused around
 * the core recurrence).  q, k, v, the decay logits a, the output gate z and the beta logits b come from one
 * packed weight matrix and are written in the layout kda_prefill_chunked reads; the causal convolution is
 * fused into the prefill's chunk kernel, which consumes these raw rows.
 *   x    device [T][hidden] bf16 hidden states (hidden % 8 == 0)
 *   w    device [N][hidden] bf16, N = H*(3*dk + 2*dv) + H: the rows of q (H*dk), k (H*dk), v (H*dv),
 *        a (H*dk), z (H*dv) and b (H), in that order (row = output feature, K-major)
 *   q, k, a  device [T][H][dk] bf16 out    v, z  device [T][H][dv] bf16 out (z may be NULL: not stored)
 *   b    device [T][H] bf16 out
 *   dev_status device int32, OR-ed with KDA_DEV_TIMEOUT if a bounded wait gave up.
 * fp32 accumulation in tensor memory; each output rounded to bf16 (nearest even).  All pointers but b
 * 16-byte aligned.  Asynchronous on `stream`; allocates nothing.
 */
KDA_API int kda_project_inputs(int64_t T, int32_t hidden, int32_t H, int32_t dk, int32_t dv, const uint16_t *x,
                               const uint16_t *w, uint16_t *q, uint16_t *k, uint16_t *v, uint16_t *a, uint16_t *b,
                               uint16_t *z, int32_t *dev_status, kda_stream_t stream);

/* Most tokens per request that one kda_decode_multi call takes. */
#define KDA_DECODE_MULTI_MAX_L 8

/*
 * L consecutive decode tokens for each of n requests in one launch, keeping the state after every position
 * on request: the verification step of speculative decoding ("vLLM Kimi K3 Support", section "Speculative
 * Decoding with DSpark": several tokens accepted per step; "moonshotai/Kimi-K3" recipe:
 * num_speculative_tokens 4, i.e. L = 5 with the bonus position).  The pages do not say how a recurrent state
 * is rolled back after a rejection; here the caller keeps the state at each position it may resume from
 * (per-position retention) and continues from the slot of the last accepted position.
 *   q, k, a   device [n*L][H][dk] bf16   v, z, y  device [n*L][H][dv] bf16   b  device [n*L][H] bf16
 *             (row r*L + j holds token j of request r; z may be NULL)
 *   src_slot  device [n] int32: state before token 0; -1 = fresh request
 *   dst_slots device [n*L] int32: the state and conv window after token j of request r go to slot
 *             dst_slots[r*L + j]; -1 = not kept.  The tokens are processed in order with the state held in
 *             fp32 between them, whatever is kept.
 *   dev_status device int32, OR-ed with KDA_DEV_* bits.
 * Each token's arithmetic is that of kda_decode_step, so L = 1 with dst_slots = dst_slot reproduces it bit
 * for bit.  Aliasing: the non-negative dst_slots of one call are distinct; a request's src may be one of its
 * own dst_slots, never another request's.  A request with a bad slot index gets y = 0 for all L tokens and
 * no state write.  1 <= L <= KDA_DECODE_MULTI_MAX_L; shapes as kda_decode_step.
 */
KDA_API int kda_decode_multi(const kda_pool *pool, const kda_params *prm, int32_t n, int32_t L, const uint16_t *q,
                             const uint16_t *k, const uint16_t *v, const uint16_t *a, const uint16_t *b,
                             const uint16_t *z, uint16_t *y, const int32_t *src_slot, const int32_t *dst_slots,
                             int32_t *dev_status, kda_stream_t stream);

/*
 * Checkpoint boundaries of one sequence: the prefix lengths p with p % interval == 0 and
 * start_pos < p <= start_pos + len ("vLLM Kimi K3 Support", section "Agentic Cache Retention Policies":
 * interval-based retention; "moonshotai/Kimi-K3" recipe: prefix-match unit 128).  Host function; returns
 * the count (0 when interval <= 0 or len <= 0), or -1 for start_pos < 0.
 */
KDA_API int64_t kda_checkpoint_count(int64_t start_pos, int64_t len, int64_t interval);

/* Bytes of device workspace kda_prefill_chunked needs for these sizes (host function, no CUDA call). */
KDA_API size_t kda_prefill_workspace_bytes(const kda_pool *pool, int32_t nseq, int64_t total_tokens, int32_t chunk);

/*
 * Chunked prefill of nseq variable-length sequences with checkpoint emission into the pool ("A Preview
 * of Production-Scale Kimi K3 Support on vLLM", sections "KDA prefill and decode" -- chunked prefill and
 * one-operation initial-state gather -- and "The Hardest Part: Prefix Caching for KDA" -- the state
 * must exist at the exact prefix boundary).
 *   cu_seqlens  device [nseq+1] int32, cu_seqlens[0] = 0, non-decreasing, cu_seqlens[nseq] = total_tokens
 *   start_pos   device [nseq] int64: absolute position of each sequence's first token (tokens already
 *               in its state); chunks are aligned to absolute positions, so a resumed sequence
 *               computes exactly what a full replay computes from the same boundary on
 *   src_slot, dst_slot  as for decode (src -1 = empty prefix)
 *   chunk       tokens per chunk (16 or 64)
 *   ckpt_interval  0 = no checkpoints; else a positive multiple of chunk
 *   ckpt_offsets   device [nseq+1] int32: sequence n's boundaries (kda_checkpoint_count of them,
 *               ascending) own entries ckpt_offsets[n] .. ckpt_offsets[n+1]-1 of ckpt_slots
 *   ckpt_slots     device int32: slot receiving (S, conv window) at that boundary, or -1 to skip.
 *               A boundary equal to the sequence end is emitted too.
 *   q,k,v,a,b,z,y  as for decode with n replaced by total_tokens (token-major)
 *   workspace   device, at least kda_prefill_workspace_bytes() bytes, contents need not be initialised
 * Same aliasing rules as decode, with checkpoint slots counting as dst slots.
 * Supported: (dk, dv) as for decode, W = 4, chunk in {16, 64}.
 * Streams: all work is ordered on `stream`.  At dk = dv = 128, chunk 64, a call with few
 * (sequence, head) chains (nseq*H*4 <= SM count) and at least 512 chunks is launched in segments.
 * The chunk chain of each segment then runs on a library-owned side stream, beside the next segment's
 * intra-chunk kernel.  The side stream forks from `stream` and joins it again before the call returns
 * (events only), so this works under CUDA graph capture too.  Segmented calls on one device are
 * serialised by a host lock.  The results are bit-identical to one launch.
 */
KDA_API int kda_prefill_chunked(const kda_pool *pool, const kda_params *prm, int32_t nseq, int64_t total_tokens,
                        const int32_t *cu_seqlens, const int64_t *start_pos, const int32_t *src_slot,
                        const int32_t *dst_slot, int32_t chunk, int64_t ckpt_interval, const int32_t *ckpt_offsets,
                        const int32_t *ckpt_slots, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                        const uint16_t *a, const uint16_t *b, const uint16_t *z, uint16_t *y, void *workspace,
                        size_t workspace_bytes, int32_t *dev_status, kda_stream_t stream);

/*
 * kda_prefill_chunked without a caller-provided workspace (the pages have no counterpart: this is an
 * interface for callers that cannot allocate device memory -- an engine whose caching allocator owns all
 * free memory, a plug-in handed only tensors, a process with no device allocation after start-up).
 * The workspace is a fixed array of KDA_NOALLOC_SCRATCH_BYTES compiled into the library; every GPU that
 * loads the library holds it until the process exits.  The call allocates nothing.
 *   Arguments: as kda_prefill_chunked, minus workspace and workspace_bytes.
 *   Limit: a problem whose kda_prefill_workspace_bytes() exceeds KDA_NOALLOC_SCRATCH_BYTES returns
 *   KDA_ERR_WORKSPACE without launching (64 MiB holds, e.g., one 512-token sequence at H = 32, dk = dv = 128).
 *   Errors: the argument checks of kda_prefill_chunked come first and make no CUDA call; then the size
 *   check (KDA_ERR_WORKSPACE); then the per-device set-up below (KDA_ERR_CUDA if it fails).
 *   Set-up: the first call on a device (with that device current) looks up the array's device address
 *   (cudaGetSymbolAddress).  Under CUDA's lazy module loading that is also when the driver allocates the
 *   array on that device, so a caller that must allocate nothing later makes this call at start-up,
 *   before it reserves its own memory pool.  The same call does the prefill launchers' one-time set-up
 *   (kernel attributes; the side stream and two events that segmented launches use), so later calls
 *   create nothing.  A call with nseq = 0 does the set-up and nothing else.  Make it before any stream
 *   capture on the device.  The address is cached per device for the life of the process; a device
 *   reset (cudaDeviceReset) invalidates it, and the library must not be used on that device afterwards.
 *   All calls on a device share the one array and it keeps the last call's contents (nothing in it needs
 *   to start at zero): calls whose executions overlap on the GPU -- on different streams, or from
 *   different host threads -- race on it and must be serialised by the caller.
 */
#define KDA_NOALLOC_SCRATCH_BYTES (64u << 20)
KDA_API int kda_prefill_chunked_noalloc(const kda_pool *pool, const kda_params *prm, int32_t nseq,
                                        int64_t total_tokens, const int32_t *cu_seqlens, const int64_t *start_pos,
                                        const int32_t *src_slot, const int32_t *dst_slot, int32_t chunk,
                                        int64_t ckpt_interval, const int32_t *ckpt_offsets,
                                        const int32_t *ckpt_slots, const uint16_t *q, const uint16_t *k,
                                        const uint16_t *v, const uint16_t *a, const uint16_t *b, const uint16_t *z,
                                        uint16_t *y, int32_t *dev_status, kda_stream_t stream);

/*
 * Copy-on-write resume ("The Hardest Part: Prefix Caching for KDA": a cached partial state is copied
 * into a private destination before the request extends it): for each of n pairs, slot dst_slot[i]
 * receives a bit-exact copy of slot src_slot[i] (state and conv window, all heads).  src_slot and
 * dst_slot are device [n] int32; dst slots must be distinct and must not be src slots of the same call.
 */
KDA_API int kda_resume_from_slot(const kda_pool *pool, int32_t n, const int32_t *src_slot, const int32_t *dst_slot,
                         int32_t *dev_status, kda_stream_t stream);

/*
 * Host-side prefix index and retention policies ("A Preview of Production-Scale Kimi K3 Support on vLLM",
 * section "The Hardest Part: Prefix Caching for KDA": chained fine-grained hashes, copy-on-write of a
 * cached partial state into a private destination, deferred same-step reuse; "vLLM Kimi K3 Support",
 * section "Agentic Cache Retention Policies": interval retention and Marconi-style second-hit retention;
 * "moonshotai/Kimi-K3" recipe: prefix-match unit 128).  Pure host code: it hands out indices of the
 * caller's state pool and fills the ckpt_slots table of kda_prefill_chunked; it allocates no device
 * memory and makes no CUDA call.  Thread-safe (one internal mutex).
 *
 * A plan for a prompt of `len` tokens:
 *   - finds the longest committed cached prefix, a multiple of the match unit shorter than the prompt;
 *   - takes a private slot for the request (copy-on-write destination; LRU-evicting an unpinned cached
 *     state when the pool is full) and pins the cached source until commit;
 *   - lists one entry per match-unit boundary p in (start_pos, len] in ckpt_slots: a slot to keep the
 *     state at p, or -1.  Call kda_prefill_chunked with ckpt_interval = the match unit, these slots,
 *     start_pos, src = private_slot and dst = private_slot, after kda_resume_from_slot(src_slot ->
 *     private_slot) when src_slot >= 0.
 * Entries a plan creates become visible to lookups only at kda_prefix_commit (after the GPU work), so a
 * request planned in the same step never resumes from a state still being written.
 */
enum kda_retention { KDA_RETAIN_INTERVAL = 0, KDA_RETAIN_SECOND_HIT = 1 };

typedef struct kda_prefix_index kda_prefix_index;

typedef struct kda_prefix_plan_t {
    uint64_t plan_id;
    int32_t src_slot;      /* cached state to resume from, or -1 */
    int32_t private_slot;  /* the request's own slot */
    int64_t start_pos;     /* tokens covered by src_slot (0 when src_slot is -1) */
    int32_t num_ckpts;     /* entries written to ckpt_slots */
    int32_t reserved;
} kda_prefix_plan_t;

/* num_slots: pool slots the index manages; match_unit: tokens per hashed block (e.g. 128);
 * interval: 0, or a multiple of match_unit (interval retention keeps multiples of it and the prompt's last
 * boundary; second-hit retention keeps seen interval boundaries and the longest seen boundary).  NULL on
 * invalid arguments. */
KDA_API kda_prefix_index *kda_prefix_index_create(int32_t num_slots, int32_t match_unit, int32_t policy,
                                                  int64_t interval);
KDA_API void kda_prefix_index_destroy(kda_prefix_index *ix);
/* Slots currently unassigned (-1 for a NULL index). */
KDA_API int32_t kda_prefix_index_free_slots(kda_prefix_index *ix);
/* tokens: host [len] int32 token ids.  ckpt_slots: host [ckpt_capacity] int32, receives num_ckpts entries.
 * KDA_ERR_INVALID_ARG for bad arguments or too small a capacity; KDA_ERR_WORKSPACE when no private slot can
 * be found (every slot pinned or pending). */
KDA_API int kda_prefix_plan(kda_prefix_index *ix, const int32_t *tokens, int64_t len, kda_prefix_plan_t *out,
                            int32_t *ckpt_slots, int32_t ckpt_capacity);
/* Publish the plan's entries and unpin its source (call once its GPU work has completed). */
KDA_API int kda_prefix_commit(kda_prefix_index *ix, uint64_t plan_id);
/* Drop an uncommitted plan: its new entries and its private slot return to the free list. */
KDA_API int kda_prefix_abort(kda_prefix_index *ix, uint64_t plan_id);
/* Return a request's private slot (not a cached state) to the free list when the request ends. */
KDA_API int kda_prefix_release_slot(kda_prefix_index *ix, int32_t slot);

/* Static description of a kda_status value. */
KDA_API const char *kda_status_string(int status);

/* What the last failing call of the calling host thread rejected ("decode: q, k, v, a and z must be
 * 16-byte aligned", "prefill launch: <CUDA error text>", ...), or "" when the last call of the thread to
 * kda_decode_step, kda_prefill_chunked(_noalloc), kda_resume_from_slot or kda_check_slots succeeded.  The
 * string belongs to the library and stays valid until the thread's next such call.  Library-side record
 * only; nothing in the pages defines it. */
KDA_API const char *kda_last_error_string(void);

/*
 * Debug check of one call's slot-aliasing contract, on HOST copies of its slot arrays.  The kernels rely
 * on it but do not check it; it is the host-side form of "same-step reuse is deferred" ("A Preview of
 * Production-Scale Kimi K3 Support on vLLM", section "The Hardest Part: Prefix Caching for KDA").
 *   - every dst_slot[i] in [0, num_slots), every src_slot[i] and ckpt_slots[j] in [-1, num_slots);
 *   - no slot is written twice: the dst slots and the non-negative checkpoint slots are distinct;
 *   - a src slot is written by nobody but its own item (src_slot[i] == dst_slot[i] is in place).
 * Decode: n_ckpt = 0.  Resume: src/dst as passed.  Prefill: its ckpt_slots table.  KDA_OK, or
 * KDA_ERR_INVALID_ARG with kda_last_error_string() naming the first violation.  O((n + n_ckpt) log), no
 * device access.
 */
KDA_API int kda_check_slots(int64_t num_slots, int32_t n, const int32_t *src_slot, const int32_t *dst_slot,
                            int32_t n_ckpt, const int32_t *ckpt_slots);

/* Failure-detection check of the bounded waits every kernel uses (no counterpart in the pages): launches
 * one CTA whose mbarrier wait can never complete; after limit_ns (clamped to [1 ms, 2 s]) of %globaltimer it
 * gives up, ORs KDA_DEV_TIMEOUT into *dev_status (device int32) and returns.  No fault, no trap: the context
 * stays usable.  Asynchronous on `stream`. */
KDA_API int kda_selftest_wait_timeout(int64_t limit_ns, int32_t *dev_status, kda_stream_t stream);

/* Library version, for the loader's sanity check. */
KDA_API int kda_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H */
