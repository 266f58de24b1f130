// kda_resume.cu -- copy-on-write of cached KDA states between pool slots ("A Preview of Production-Scale
// Kimi K3 Support on vLLM", section "The Hardest Part: Prefix Caching for KDA": a cached partial state
// is copied into a private destination before the request extends it).
//
// Pure bandwidth: one CTA per (pair, head) moves the fp32 state and the bf16 window with 128-bit
// loads issued back to back (all loads of a thread in flight before its first store).  Bit-exact.
#include "kda_device.cuh"
#include "kda_internal.h"

namespace kda {

constexpr int kResumeThreads = 256;
constexpr int kResumeUnroll = 16;  // 16-byte words per thread per round

__global__ void __launch_bounds__(kResumeThreads) kda_resume_kernel(const ResumeArgs a) {
    const int pair = blockIdx.x / a.H, h = blockIdx.x - (blockIdx.x / a.H) * a.H;
    const int src = a.src[pair], dst = a.dst[pair];
    if (src < 0 || src >= a.num_slots || dst < 0 || dst >= a.num_slots) {
        if (threadIdx.x == 0) set_status(a.status, KDA_DEV_BAD_SLOT);
        return;
    }
    const uint4 *sS = reinterpret_cast<const uint4 *>(a.S) + ((size_t)src * a.H + h) * a.s_words16;
    uint4 *dS = reinterpret_cast<uint4 *>(a.S) + ((size_t)dst * a.H + h) * a.s_words16;
    for (int base = 0; base < a.s_words16; base += kResumeThreads * kResumeUnroll) {
        uint4 r[kResumeUnroll];
#pragma unroll
        for (int u = 0; u < kResumeUnroll; ++u) {
            const int i = base + u * kResumeThreads + threadIdx.x;
            if (i < a.s_words16) r[u] = __ldcs(sS + i);
        }
#pragma unroll
        for (int u = 0; u < kResumeUnroll; ++u) {
            const int i = base + u * kResumeThreads + threadIdx.x;
            if (i < a.s_words16) dS[i] = r[u];
        }
    }
    const uint4 *sC = reinterpret_cast<const uint4 *>(a.conv) + ((size_t)src * a.H + h) * a.conv_words16;
    uint4 *dC = reinterpret_cast<uint4 *>(a.conv) + ((size_t)dst * a.H + h) * a.conv_words16;
    for (int i = threadIdx.x; i < a.conv_words16; i += kResumeThreads) dC[i] = sC[i];
}

int launch_resume(const ResumeArgs &a, cudaStream_t st) {
    const long long blocks = (long long)a.n * a.H;
    if (blocks > 0x7fffffffLL) return fail(KDA_ERR_INVALID_ARG, "resume: n * H too large");
    kda_resume_kernel<<<(unsigned)blocks, kResumeThreads, 0, st>>>(a);
    return launch_result("kda_resume_kernel launch");
}

}  // namespace kda
