// kda_internal.h -- launcher interfaces between the C-ABI layer (kda_api.cu) and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/kda.h"

namespace kda {

struct DecodeArgs {
    void *S;             // pool states [num_slots][H][dk][dv], fp32 or bf16 (state_bf16)
    int32_t state_bf16;
    uint16_t *conv;      // pool windows [num_slots][H][W-1][2dk+dv]
    int64_t num_slots;
    int32_t H, n;
    const float *conv_w, *norm_w;
    float l2_eps, rms_eps, scale;
    int32_t silu;
    const uint16_t *q, *k, *v, *a, *b, *z;
    uint16_t *y;
    const int32_t *src, *dst;
    int32_t *status;
};

struct ResumeArgs {
    void *S;
    uint16_t *conv;
    int64_t num_slots;
    int32_t H, n;
    int32_t s_words16;     // 16-byte words per (slot, head) state
    int32_t conv_words16;  // 16-byte words per (slot, head) window
    const int32_t *src, *dst;
    int32_t *status;
};

struct PrefillArgs {
    void *S;             // fp32 or bf16 (state_bf16)
    int32_t state_bf16;
    uint16_t *conv;
    int64_t num_slots;
    int32_t H, nseq;
    int64_t total_tokens;
    const float *conv_w, *norm_w;
    float l2_eps, rms_eps, scale;
    int32_t silu;
    const int32_t *cu_seqlens;
    const int64_t *start_pos;
    const int32_t *src, *dst;
    int32_t chunk;
    int64_t interval;
    const int32_t *ckpt_offsets, *ckpt_slots;
    const uint16_t *q, *k, *v, *a, *b, *z;
    uint16_t *y;
    void *ws;
    size_t ws_bytes;
    int32_t *status;
    // Range [seg_lo, seg_hi) of the call's chunks (numbered over all sequences) that one launch of the
    // tensor-core kernels processes; the whole call unless the launcher splits it into segments.
    int32_t seg_lo = 0, seg_hi = INT32_MAX;
};

bool decode_supported(int dk, int dv, int W);
int launch_decode(const DecodeArgs &a, int dk, int dv, cudaStream_t st);
// L tokens per request; a.dst is the [n*L] table of kept positions (-1 = not kept).
int launch_decode_multi(const DecodeArgs &a, int dk, int dv, int L, cudaStream_t st);

int launch_resume(const ResumeArgs &a, cudaStream_t st);

struct ProjectArgs {
    int64_t T;
    int32_t hidden, H, dk, dv;
    const uint16_t *x, *w;                 // [T][hidden], [N][hidden] bf16
    uint16_t *q, *k, *v, *a, *z, *b;       // [T][H][dk | dv], b [T][H]; z may be NULL
    int32_t *status;
};
int launch_project(const ProjectArgs &a, cudaStream_t st);

bool prefill_supported(int dk, int dv, int W, int chunk);
// The host-side argument checks of kda_prefill_chunked (everything but the workspace); KDA_OK or the failure
// code with the reason recorded.  Makes no CUDA call.
int check_prefill_args(const kda_pool *pool, const kda_params *prm, int32_t nseq, int64_t total_tokens,
                       const int32_t *cu_seqlens, const int64_t *start_pos, const int32_t *src_slot,
                       const int32_t *dst_slot, int32_t chunk, int64_t ckpt_interval, const int32_t *ckpt_offsets,
                       const int32_t *ckpt_slots, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                       const uint16_t *a, const uint16_t *b, const uint16_t *z, const uint16_t *y,
                       const int32_t *dev_status);
// One-time per-device set-up of the prefill launchers, done on the current device: kernel attributes, the
// tensor-map encoder, the SM count, and the side stream and events of segmented launches.  Later calls do
// nothing.  KDA_OK or KDA_ERR_CUDA.
int prefill_prepare();
size_t prefill_workspace_bytes(int H, int dk, int dv, int nseq, int64_t total_tokens, int chunk);
int launch_prefill(const PrefillArgs &a, int dk, int dv, cudaStream_t st);

// Streaming multiprocessors of the current device (cached per device).
int current_device_sms();

// Per-host-thread description of the most recent failure, read by kda_last_error_string().
// fail() records `what` and returns `code`; clear_error() runs at the start of every entry point.
int fail(int code, const char *what);
void clear_error();
// KDA_OK if the launches just issued were accepted; else KDA_ERR_CUDA with "<what>: <CUDA error>" recorded.
int launch_result(const char *what);

}  // namespace kda
