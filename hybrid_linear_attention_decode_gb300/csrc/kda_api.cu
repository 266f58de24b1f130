// kda_api.cu -- the C ABI (include/kda.h): argument validation, dispatch to the kernel launchers.
// No allocation, no host synchronisation, no global state beyond per-device attribute caches and the
// per-thread description of the last failure.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <vector>

#include "../../include/kda.h"
#include "kda_internal.h"

namespace kda {

static thread_local char t_last_error[320] = "";

int fail(int code, const char *what) {
    snprintf(t_last_error, sizeof(t_last_error), "%s", what ? what : "");
    return code;
}

void clear_error() { t_last_error[0] = '\0'; }

int launch_result(const char *what) {
    const cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) return KDA_OK;
    snprintf(t_last_error, sizeof(t_last_error), "%s: %s", what, cudaGetErrorString(e));
    return KDA_ERR_CUDA;
}

int current_device_sms() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
    if (cache[dev] == 0) {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1) sms = 1;
        cache[dev] = sms;
    }
    return cache[dev];
}

static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
static bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
static bool aligned2(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 1u) == 0; }

static int check_pool(const kda_pool *pool, const kda_params *prm) {
    if (!pool) return fail(KDA_ERR_INVALID_ARG, "pool is NULL");
    if (!pool->S || !pool->conv) return fail(KDA_ERR_INVALID_ARG, "pool->S or pool->conv is NULL");
    if (pool->H <= 0 || pool->num_slots <= 0 || pool->dk <= 0 || pool->dv <= 0)
        return fail(KDA_ERR_INVALID_ARG, "pool H, dk, dv and num_slots must be positive");
    if (pool->state_dtype != KDA_STATE_FP32 && pool->state_dtype != KDA_STATE_BF16)
        return fail(KDA_ERR_INVALID_ARG, "pool->state_dtype is neither KDA_STATE_FP32 nor KDA_STATE_BF16");
    if (!aligned16(pool->S) || !aligned16(pool->conv))
        return fail(KDA_ERR_INVALID_ARG, "pool->S and pool->conv must be 16-byte aligned");
    if (prm) {
        if (!prm->conv_weight || !prm->norm_weight)
            return fail(KDA_ERR_INVALID_ARG, "params conv_weight or norm_weight is NULL");
        if (!aligned16(prm->conv_weight) || !aligned4(prm->norm_weight))
            return fail(KDA_ERR_INVALID_ARG, "conv_weight must be 16-byte and norm_weight 4-byte aligned");
        if (!(prm->l2_eps >= 0.f) || !(prm->rms_eps >= 0.f))
            return fail(KDA_ERR_INVALID_ARG, "l2_eps and rms_eps must be >= 0");
    }
    return KDA_OK;
}

int check_prefill_args(const kda_pool *pool, const kda_params *prm, int32_t nseq, int64_t total_tokens,
                       const int32_t *cu_seqlens, const int64_t *start_pos, const int32_t *src_slot,
                       const int32_t *dst_slot, int32_t chunk, int64_t ckpt_interval, const int32_t *ckpt_offsets,
                       const int32_t *ckpt_slots, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                       const uint16_t *a, const uint16_t *b, const uint16_t *z, const uint16_t *y,
                       const int32_t *dev_status) {
    int rc = check_pool(pool, prm);
    if (rc != KDA_OK) return rc;
    if (!prm) return fail(KDA_ERR_INVALID_ARG, "prefill: params is NULL");
    if (nseq < 0 || total_tokens < 0 || ckpt_interval < 0)
        return fail(KDA_ERR_INVALID_ARG, "prefill: nseq, total_tokens and ckpt_interval must be >= 0");
    if (!prefill_supported(pool->dk, pool->dv, pool->conv_w, chunk))
        return fail(KDA_ERR_UNSUPPORTED_SHAPE, "prefill: (dk, dv, conv_w, chunk) not compiled in");
    if (ckpt_interval > 0 && ckpt_interval % chunk != 0)
        return fail(KDA_ERR_INVALID_ARG, "prefill: ckpt_interval is not a multiple of the chunk");
    if (nseq == 0) return KDA_OK;
    if (!cu_seqlens || !start_pos || !src_slot || !dst_slot)
        return fail(KDA_ERR_INVALID_ARG, "prefill: cu_seqlens, start_pos, src_slot or dst_slot is NULL");
    if (ckpt_interval > 0 && (!ckpt_offsets || !ckpt_slots))
        return fail(KDA_ERR_INVALID_ARG, "prefill: checkpoints requested without ckpt_offsets / ckpt_slots");
    if (total_tokens > 0 && (!q || !k || !v || !a || !b || !y))
        return fail(KDA_ERR_INVALID_ARG, "prefill: a token tensor is NULL");
    if (total_tokens * (int64_t)pool->H > ((int64_t)1 << 40))
        return fail(KDA_ERR_INVALID_ARG, "prefill: total_tokens * H too large");
    if ((q && !aligned16(q)) || (k && !aligned16(k)) || (v && !aligned16(v)) || (a && !aligned16(a)) ||
        (z && !aligned16(z)) || (y && !aligned16(y)))
        return fail(KDA_ERR_INVALID_ARG, "prefill: q, k, v, a, z and y must be 16-byte aligned");
    if ((b && !aligned2(b)) || !aligned4(cu_seqlens) || (reinterpret_cast<uintptr_t>(start_pos) & 7u) ||
        !aligned4(src_slot) || !aligned4(dst_slot) || (dev_status && !aligned4(dev_status)))
        return fail(KDA_ERR_INVALID_ARG, "prefill: b, tables, slot arrays or status misaligned");
    return KDA_OK;
}

}  // namespace kda

using namespace kda;

extern "C" {

int kda_version(void) { return 1; }

const char *kda_status_string(int status) {
    switch (status) {
        case KDA_OK: return "ok";
        case KDA_ERR_INVALID_ARG: return "invalid argument (null, negative, misaligned or inconsistent)";
        case KDA_ERR_UNSUPPORTED_SHAPE: return "unsupported shape (dk, dv, conv width or chunk)";
        case KDA_ERR_WORKSPACE: return "workspace missing or too small";
        case KDA_ERR_CUDA: return "CUDA launch or attribute call failed";
        default: return "unknown status";
    }
}

const char *kda_last_error_string(void) { return t_last_error; }

int64_t kda_checkpoint_count(int64_t start_pos, int64_t len, int64_t interval) {
    if (start_pos < 0) return -1;
    if (interval <= 0 || len <= 0) return 0;
    return (start_pos + len) / interval - start_pos / interval;
}

int kda_check_slots(int64_t num_slots, int32_t n, const int32_t *src_slot, const int32_t *dst_slot, int32_t n_ckpt,
                    const int32_t *ckpt_slots) {
    clear_error();
    char msg[160];
    if (num_slots <= 0 || n < 0 || n_ckpt < 0 || (n > 0 && (!src_slot || !dst_slot)) || (n_ckpt > 0 && !ckpt_slots))
        return fail(KDA_ERR_INVALID_ARG, "check_slots: bad counts or NULL arrays");
    std::vector<int64_t> written;  // every slot the call writes: the dst slots and the kept checkpoints
    written.reserve((size_t)n + (size_t)n_ckpt);
    for (int32_t i = 0; i < n; ++i) {
        const int32_t d = dst_slot[i], s = src_slot[i];
        if (d < 0 || d >= num_slots) {
            snprintf(msg, sizeof(msg), "check_slots: dst_slot[%d] = %d outside [0, %lld)", i, d, (long long)num_slots);
            return fail(KDA_ERR_INVALID_ARG, msg);
        }
        if (s < -1 || s >= num_slots) {
            snprintf(msg, sizeof(msg), "check_slots: src_slot[%d] = %d outside [-1, %lld)", i, s, (long long)num_slots);
            return fail(KDA_ERR_INVALID_ARG, msg);
        }
        written.push_back(d);
    }
    for (int32_t j = 0; j < n_ckpt; ++j) {
        const int32_t c = ckpt_slots[j];
        if (c < -1 || c >= num_slots) {
            snprintf(msg, sizeof(msg), "check_slots: ckpt_slots[%d] = %d outside [-1, %lld)", j, c, (long long)num_slots);
            return fail(KDA_ERR_INVALID_ARG, msg);
        }
        if (c >= 0) written.push_back(c);
    }
    std::vector<int64_t> sorted_w(written);
    std::sort(sorted_w.begin(), sorted_w.end());
    for (size_t i = 1; i < sorted_w.size(); ++i)
        if (sorted_w[i] == sorted_w[i - 1]) {
            snprintf(msg, sizeof(msg), "check_slots: slot %lld is written twice (dst or checkpoint)",
                     (long long)sorted_w[i]);
            return fail(KDA_ERR_INVALID_ARG, msg);
        }
    // a src may only coincide with its own item's dst (in place; a second write of that slot is a duplicate)
    for (int32_t i = 0; i < n; ++i) {
        const int32_t s = src_slot[i];
        if (s < 0 || s == dst_slot[i]) continue;
        if (std::binary_search(sorted_w.begin(), sorted_w.end(), (int64_t)s)) {
            snprintf(msg, sizeof(msg), "check_slots: src_slot[%d] = %d is written by another item or a checkpoint",
                     i, s);
            return fail(KDA_ERR_INVALID_ARG, msg);
        }
    }
    return KDA_OK;
}

int kda_decode_step(const kda_pool *pool, const kda_params *prm, int32_t n, const uint16_t *q, const uint16_t *k,
                    const uint16_t *v, const uint16_t *a, const uint16_t *b, const uint16_t *z, uint16_t *y,
                    const int32_t *src_slot, const int32_t *dst_slot, int32_t *dev_status, kda_stream_t stream) {
    clear_error();
    int rc = check_pool(pool, prm);
    if (rc != KDA_OK) return rc;
    if (!prm) return fail(KDA_ERR_INVALID_ARG, "decode: params is NULL");
    if (n < 0) return fail(KDA_ERR_INVALID_ARG, "decode: n < 0");
    if (!decode_supported(pool->dk, pool->dv, pool->conv_w))
        return fail(KDA_ERR_UNSUPPORTED_SHAPE, "decode: (dk, dv, conv_w) not compiled in");
    if (n == 0) return KDA_OK;
    if ((int64_t)n * pool->H > 0x7fffffffLL) return fail(KDA_ERR_INVALID_ARG, "decode: n * H too large");
    if (!q || !k || !v || !a || !b || !y || !src_slot || !dst_slot)
        return fail(KDA_ERR_INVALID_ARG, "decode: a required pointer is NULL");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(a) || (z && !aligned16(z)))
        return fail(KDA_ERR_INVALID_ARG, "decode: q, k, v, a and z must be 16-byte aligned");
    if (!aligned2(b) || !aligned2(y) || !aligned4(src_slot) || !aligned4(dst_slot) ||
        (dev_status && !aligned4(dev_status)))
        return fail(KDA_ERR_INVALID_ARG, "decode: b, y, slot arrays or status misaligned");
    DecodeArgs d;
    d.S = pool->S;
    d.state_bf16 = pool->state_dtype == KDA_STATE_BF16;
    d.conv = pool->conv;
    d.num_slots = pool->num_slots;
    d.H = pool->H;
    d.n = n;
    d.conv_w = prm->conv_weight;
    d.norm_w = prm->norm_weight;
    d.l2_eps = prm->l2_eps;
    d.rms_eps = prm->rms_eps;
    d.scale = prm->scale;
    d.silu = prm->conv_silu;
    d.q = q; d.k = k; d.v = v; d.a = a; d.b = b; d.z = z; d.y = y;
    d.src = src_slot;
    d.dst = dst_slot;
    d.status = dev_status;
    return launch_decode(d, pool->dk, pool->dv, reinterpret_cast<cudaStream_t>(stream));
}

int kda_decode_multi(const kda_pool *pool, const kda_params *prm, int32_t n, int32_t L, const uint16_t *q,
                     const uint16_t *k, const uint16_t *v, const uint16_t *a, const uint16_t *b, const uint16_t *z,
                     uint16_t *y, const int32_t *src_slot, const int32_t *dst_slots, int32_t *dev_status,
                     kda_stream_t stream) {
    clear_error();
    int rc = check_pool(pool, prm);
    if (rc != KDA_OK) return rc;
    if (!prm) return fail(KDA_ERR_INVALID_ARG, "decode_multi: params is NULL");
    if (n < 0) return fail(KDA_ERR_INVALID_ARG, "decode_multi: n < 0");
    if (L < 1 || L > KDA_DECODE_MULTI_MAX_L)
        return fail(KDA_ERR_INVALID_ARG, "decode_multi: L outside [1, KDA_DECODE_MULTI_MAX_L]");
    if (!decode_supported(pool->dk, pool->dv, pool->conv_w))
        return fail(KDA_ERR_UNSUPPORTED_SHAPE, "decode_multi: (dk, dv, conv_w) not compiled in");
    if (n == 0) return KDA_OK;
    if ((int64_t)n * L * pool->H > 0x7fffffffLL) return fail(KDA_ERR_INVALID_ARG, "decode_multi: n * L * H too large");
    if (!q || !k || !v || !a || !b || !y || !src_slot || !dst_slots)
        return fail(KDA_ERR_INVALID_ARG, "decode_multi: a required pointer is NULL");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(a) || (z && !aligned16(z)))
        return fail(KDA_ERR_INVALID_ARG, "decode_multi: q, k, v, a and z must be 16-byte aligned");
    if (!aligned2(b) || !aligned2(y) || !aligned4(src_slot) || !aligned4(dst_slots) ||
        (dev_status && !aligned4(dev_status)))
        return fail(KDA_ERR_INVALID_ARG, "decode_multi: b, y, slot arrays or status misaligned");
    DecodeArgs d;
    d.S = pool->S;
    d.state_bf16 = pool->state_dtype == KDA_STATE_BF16;
    d.conv = pool->conv;
    d.num_slots = pool->num_slots;
    d.H = pool->H;
    d.n = n;
    d.conv_w = prm->conv_weight;
    d.norm_w = prm->norm_weight;
    d.l2_eps = prm->l2_eps;
    d.rms_eps = prm->rms_eps;
    d.scale = prm->scale;
    d.silu = prm->conv_silu;
    d.q = q; d.k = k; d.v = v; d.a = a; d.b = b; d.z = z; d.y = y;
    d.src = src_slot;
    d.dst = dst_slots;
    d.status = dev_status;
    return launch_decode_multi(d, pool->dk, pool->dv, L, reinterpret_cast<cudaStream_t>(stream));
}

int kda_project_inputs(int64_t T, int32_t hidden, int32_t H, int32_t dk, int32_t dv, const uint16_t *x,
                       const uint16_t *w, uint16_t *q, uint16_t *k, uint16_t *v, uint16_t *a, uint16_t *b, uint16_t *z,
                       int32_t *dev_status, kda_stream_t stream) {
    clear_error();
    if (T < 0 || hidden <= 0 || H <= 0 || dk <= 0 || dv <= 0)
        return fail(KDA_ERR_INVALID_ARG, "project: T must be >= 0 and hidden, H, dk, dv positive");
    if (hidden % 8) return fail(KDA_ERR_INVALID_ARG, "project: hidden must be a multiple of 8 (16-byte rows)");
    if (T > 0x7fffffffLL || (int64_t)H * (3 * dk + 2 * dv + 1) > 0x7fffffffLL)
        return fail(KDA_ERR_INVALID_ARG, "project: T or the projection width too large");
    if (T == 0) return KDA_OK;
    if (!x || !w || !q || !k || !v || !a || !b) return fail(KDA_ERR_INVALID_ARG, "project: a required pointer is NULL");
    if (!aligned16(x) || !aligned16(w) || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(a) ||
        (z && !aligned16(z)) || !aligned2(b) || (dev_status && !aligned4(dev_status)))
        return fail(KDA_ERR_INVALID_ARG, "project: x, w, q, k, v, a, z must be 16-byte aligned, b 2-byte");
    ProjectArgs p;
    p.T = T;
    p.hidden = hidden;
    p.H = H;
    p.dk = dk;
    p.dv = dv;
    p.x = x; p.w = w;
    p.q = q; p.k = k; p.v = v; p.a = a; p.z = z; p.b = b;
    p.status = dev_status;
    return launch_project(p, reinterpret_cast<cudaStream_t>(stream));
}

size_t kda_prefill_workspace_bytes(const kda_pool *pool, int32_t nseq, int64_t total_tokens, int32_t chunk) {
    if (!pool || nseq < 0 || total_tokens < 0 || pool->H <= 0) return 0;
    if (!prefill_supported(pool->dk, pool->dv, pool->conv_w, chunk)) return 0;
    return prefill_workspace_bytes(pool->H, pool->dk, pool->dv, nseq, total_tokens, chunk);
}

int kda_prefill_chunked(const kda_pool *pool, const kda_params *prm, int32_t nseq, int64_t total_tokens,
                        const int32_t *cu_seqlens, const int64_t *start_pos, const int32_t *src_slot,
                        const int32_t *dst_slot, int32_t chunk, int64_t ckpt_interval, const int32_t *ckpt_offsets,
                        const int32_t *ckpt_slots, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                        const uint16_t *a, const uint16_t *b, const uint16_t *z, uint16_t *y, void *workspace,
                        size_t workspace_bytes, int32_t *dev_status, kda_stream_t stream) {
    clear_error();
    const int rc = check_prefill_args(pool, prm, nseq, total_tokens, cu_seqlens, start_pos, src_slot, dst_slot, chunk,
                                      ckpt_interval, ckpt_offsets, ckpt_slots, q, k, v, a, b, z, y, dev_status);
    if (rc != KDA_OK || nseq == 0) return rc;
    const size_t need = prefill_workspace_bytes(pool->H, pool->dk, pool->dv, nseq, total_tokens, chunk);
    if (!workspace || workspace_bytes < need || !aligned16(workspace))
        return fail(KDA_ERR_WORKSPACE, "prefill: workspace NULL, misaligned or smaller than "
                                       "kda_prefill_workspace_bytes()");
    PrefillArgs p;
    p.S = pool->S;
    p.state_bf16 = pool->state_dtype == KDA_STATE_BF16;
    p.conv = pool->conv;
    p.num_slots = pool->num_slots;
    p.H = pool->H;
    p.nseq = nseq;
    p.total_tokens = total_tokens;
    p.conv_w = prm->conv_weight;
    p.norm_w = prm->norm_weight;
    p.l2_eps = prm->l2_eps;
    p.rms_eps = prm->rms_eps;
    p.scale = prm->scale;
    p.silu = prm->conv_silu;
    p.cu_seqlens = cu_seqlens;
    p.start_pos = start_pos;
    p.src = src_slot;
    p.dst = dst_slot;
    p.chunk = chunk;
    p.interval = ckpt_interval;
    p.ckpt_offsets = ckpt_offsets;
    p.ckpt_slots = ckpt_slots;
    p.q = q; p.k = k; p.v = v; p.a = a; p.b = b; p.z = z; p.y = y;
    p.ws = workspace;
    p.ws_bytes = workspace_bytes;
    p.status = dev_status;
    return launch_prefill(p, pool->dk, pool->dv, reinterpret_cast<cudaStream_t>(stream));
}

int kda_resume_from_slot(const kda_pool *pool, int32_t n, const int32_t *src_slot, const int32_t *dst_slot,
                         int32_t *dev_status, kda_stream_t stream) {
    clear_error();
    int rc = check_pool(pool, nullptr);
    if (rc != KDA_OK) return rc;
    if (n < 0) return fail(KDA_ERR_INVALID_ARG, "resume: n < 0");
    if (n == 0) return KDA_OK;
    if (!src_slot || !dst_slot || !aligned4(src_slot) || !aligned4(dst_slot))
        return fail(KDA_ERR_INVALID_ARG, "resume: slot arrays NULL or misaligned");
    if (pool->conv_w < 1) return fail(KDA_ERR_INVALID_ARG, "resume: conv_w < 1");
    const int64_t s_bytes = (int64_t)pool->dk * pool->dv * (pool->state_dtype == KDA_STATE_BF16 ? 2 : 4);
    const int64_t c_bytes = (int64_t)(pool->conv_w - 1) * (2 * pool->dk + pool->dv) * 2;
    if (s_bytes % 16 || c_bytes % 16)
        return fail(KDA_ERR_UNSUPPORTED_SHAPE, "resume: state or window size not a multiple of 16 bytes");
    ResumeArgs r;
    r.S = pool->S;
    r.conv = pool->conv;
    r.num_slots = pool->num_slots;
    r.H = pool->H;
    r.n = n;
    r.s_words16 = (int32_t)(s_bytes / 16);
    r.conv_words16 = (int32_t)(c_bytes / 16);
    r.src = src_slot;
    r.dst = dst_slot;
    r.status = dev_status;
    return launch_resume(r, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
