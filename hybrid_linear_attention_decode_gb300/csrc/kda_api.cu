// kda_api.cu -- the C ABI (include/kda.h): argument validation, dispatch to the kernel launchers.
// No allocation, no host synchronisation, no global state beyond per-device attribute caches.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kda.h"
#include "kda_internal.h"

namespace kda {

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
    if (!pool || !pool->S || !pool->conv || pool->H <= 0 || pool->num_slots <= 0 || pool->dk <= 0 || pool->dv <= 0)
        return KDA_ERR_INVALID_ARG;
    if (pool->state_dtype != KDA_STATE_FP32 && pool->state_dtype != KDA_STATE_BF16) return KDA_ERR_INVALID_ARG;
    if (!aligned16(pool->S) || !aligned16(pool->conv)) return KDA_ERR_INVALID_ARG;
    if (prm) {
        if (!prm->conv_weight || !prm->norm_weight) return KDA_ERR_INVALID_ARG;
        if (!aligned16(prm->conv_weight) || !aligned4(prm->norm_weight)) return KDA_ERR_INVALID_ARG;
        if (!(prm->l2_eps >= 0.f) || !(prm->rms_eps >= 0.f)) return KDA_ERR_INVALID_ARG;
    }
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

int64_t kda_checkpoint_count(int64_t start_pos, int64_t len, int64_t interval) {
    if (start_pos < 0) return -1;
    if (interval <= 0 || len <= 0) return 0;
    return (start_pos + len) / interval - start_pos / interval;
}

int kda_decode_step(const kda_pool *pool, const kda_params *prm, int32_t n, const uint16_t *q, const uint16_t *k,
                    const uint16_t *v, const uint16_t *a, const uint16_t *b, const uint16_t *z, uint16_t *y,
                    const int32_t *src_slot, const int32_t *dst_slot, int32_t *dev_status, kda_stream_t stream) {
    int rc = check_pool(pool, prm);
    if (rc != KDA_OK) return rc;
    if (!prm || n < 0) return KDA_ERR_INVALID_ARG;
    if (!decode_supported(pool->dk, pool->dv, pool->conv_w)) return KDA_ERR_UNSUPPORTED_SHAPE;
    if (n == 0) return KDA_OK;
    if ((int64_t)n * pool->H > 0x7fffffffLL) return KDA_ERR_INVALID_ARG;
    if (!q || !k || !v || !a || !b || !y || !src_slot || !dst_slot) return KDA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(a) || (z && !aligned16(z)) || !aligned2(b) ||
        !aligned2(y) || !aligned4(src_slot) || !aligned4(dst_slot) || (dev_status && !aligned4(dev_status)))
        return KDA_ERR_INVALID_ARG;
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
    int rc = check_pool(pool, prm);
    if (rc != KDA_OK) return rc;
    if (!prm || nseq < 0 || total_tokens < 0 || ckpt_interval < 0) return KDA_ERR_INVALID_ARG;
    if (!prefill_supported(pool->dk, pool->dv, pool->conv_w, chunk)) return KDA_ERR_UNSUPPORTED_SHAPE;
    if (ckpt_interval > 0 && ckpt_interval % chunk != 0) return KDA_ERR_INVALID_ARG;
    if (nseq == 0) return KDA_OK;
    if (!cu_seqlens || !start_pos || !src_slot || !dst_slot) return KDA_ERR_INVALID_ARG;
    if (ckpt_interval > 0 && (!ckpt_offsets || !ckpt_slots)) return KDA_ERR_INVALID_ARG;
    if (total_tokens > 0 && (!q || !k || !v || !a || !b || !y)) return KDA_ERR_INVALID_ARG;
    if (total_tokens * (int64_t)pool->H > ((int64_t)1 << 40)) return KDA_ERR_INVALID_ARG;
    if ((q && !aligned16(q)) || (k && !aligned16(k)) || (v && !aligned16(v)) || (a && !aligned16(a)) ||
        (z && !aligned16(z)) || (b && !aligned2(b)) || (y && !aligned16(y)) || !aligned4(cu_seqlens) ||
        (reinterpret_cast<uintptr_t>(start_pos) & 7u) || !aligned4(src_slot) || !aligned4(dst_slot) ||
        (dev_status && !aligned4(dev_status)))
        return KDA_ERR_INVALID_ARG;
    const size_t need = prefill_workspace_bytes(pool->H, pool->dk, pool->dv, nseq, total_tokens, chunk);
    if (!workspace || workspace_bytes < need || !aligned16(workspace)) return KDA_ERR_WORKSPACE;
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
    int rc = check_pool(pool, nullptr);
    if (rc != KDA_OK) return rc;
    if (n < 0) return KDA_ERR_INVALID_ARG;
    if (n == 0) return KDA_OK;
    if (!src_slot || !dst_slot || !aligned4(src_slot) || !aligned4(dst_slot)) return KDA_ERR_INVALID_ARG;
    if (pool->conv_w < 1) return KDA_ERR_INVALID_ARG;
    const int64_t s_bytes = (int64_t)pool->dk * pool->dv * (pool->state_dtype == KDA_STATE_BF16 ? 2 : 4);
    const int64_t c_bytes = (int64_t)(pool->conv_w - 1) * (2 * pool->dk + pool->dv) * 2;
    if (s_bytes % 16 || c_bytes % 16) return KDA_ERR_UNSUPPORTED_SHAPE;
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
