// Host-side context of the HSQ library and the helpers shared by the
// translation units that launch kernels (hsq_kernels.cu, hsq_decode_r*.cu).
#pragma once

#include <cuda_runtime.h>

#include <string>
#include <vector>

#include "hsq_internal.h"

struct hsq_ctx {
    hsq_config cfg;
    int r = 1, num_sms = 0, device = 0, smem_optin = 0;
    int G_max = 0, W_max = 0;
    float* d_cb = nullptr;
    float* d_rope_hi = nullptr;
    float* d_rope_lo = nullptr;
    float* d_scores = nullptr;
    int* d_route_ctr = nullptr;
    int* d_prefix = nullptr;
    int* d_err = nullptr;
    float* d_qjl_sb = nullptr;  // TQ-QKV: the last encode's S Pi as tensor-core B fragments (64 KB)
    // TQ-QKV: the last encode's L3 key codes and norms in device memory,
    // [max_batch][Hkv][G_max][N * 64 codes | N f32 norms], read by the sketch pass
    uint8_t* d_qjl_kc = nullptr;
    // Decode launch plan per cache shape: cluster size S (0 = no launchable
    // shape) and whether the split's inputs are staged in shared memory.
    struct Plan { int B, T, route, S, staged; };
    std::vector<Plan> plans;
    std::vector<const void*> accessible;  // caller pointers already checked (device or mapped host)
    std::string last_error;
};

namespace hsq {

// Records msg as the context's (and the process's) last error; returns st.
hsq_status fail(hsq_ctx* ctx, hsq_status st, const std::string& msg);
hsq_status cuda_fail(hsq_ctx* ctx, cudaError_t e, const char* where);

// Process-wide, raise-only dynamic shared-memory limit of a kernel on a device.
cudaError_t raise_smem_limit(const void* fn, int device, size_t bytes);
// Allows 16-CTA clusters for a kernel on a device (once).
cudaError_t allow_big_clusters(const void* fn, int device);

// Decode step of one layer for head ratio r = Hq / Hkv (hsq_decode_r<r>.cu).
// route: select (hsq_decode_step) or read sel (hsq_decode_attn).  *launched
// is false when no cluster shape can be launched for this cache (nothing
// was enqueued, HSQ_OK returned).
#define HSQ_DECLARE_DECODE(R)                                                                          \
    hsq_status decode_run_r##R(hsq_ctx* ctx, const hsq_cache* cache, const float* q, const int32_t* pos, \
                               int32_t* sel, float* out, bool route, bool from_staging, cudaStream_t st,  \
                               bool* launched);
HSQ_DECLARE_DECODE(1)
HSQ_DECLARE_DECODE(2)
HSQ_DECLARE_DECODE(4)
HSQ_DECLARE_DECODE(5)
HSQ_DECLARE_DECODE(8)
#undef HSQ_DECLARE_DECODE

// Prefill (hsq_prefill.cu): the attention operands as shared-memory images in
// the caller's workspace (layout in hsq_prefill.cu) and the kernels around them.
struct PrefillImages {
    uint8_t *qh, *ql, *kh, *kl, *vt;
    int nqt, nkt;   // 128-query tiles, 64-key tiles (2 nqt)
    size_t bytes;   // workspace bytes the images take
};
PrefillImages prefill_images(void* ws, int B, int Hq, int Hkv, int T);
hsq_status prefill_prep_q(hsq_ctx* ctx, const PrefillImages& im, const void* Q, int B, int T, cudaStream_t st);
hsq_status prefill_prep_kv(hsq_ctx* ctx, const PrefillImages& im, const void* K, const void* V, int B, int T,
                           cudaStream_t st);
hsq_status prefill_attention(hsq_ctx* ctx, const PrefillImages& im, float* out, int B, int T, cudaStream_t st);

}  // namespace hsq
