// HSQ compressed-KV kernels for GB300 (sm_103a) and the C entry points that
// launch them.
//
// Method: Tamarin (HSQ) technical summary (gist.science rs-10297225),
// section 2: three-tier cache (L1 focal 4-bit, L2 3-bit group summaries,
// L3 4-bit archive) and the decode process (route -> fetch + dequantise +
// rotate to position -> attention over the union, fetched summaries
// masked).  TurboQuant: "Ablation, Statistical Inference, and Validation
// for KV-Cache Compression" (gist.science 2607.09683), experimental setup
// item 1 (randomised Walsh-Hadamard transform + Beta Lloyd-Max codebook).
//
// Thread mapping.  Every 128-d vector is handled by one half-warp (16
// lanes).  Lane l of the half holds dims {4l..4l+3} in v[0..3] and
// {64+4l..64+4l+3} in v[4..7]:
//   * RoPE pairs (i, i+64) sit in the same lane, so RoPE needs no shuffle;
//   * the Walsh-Hadamard transform runs its index bits 0, 1 and 6 in
//     registers and bits 2-5 as four xor-shuffles inside the half-warp;
//   * 4-bit codes of a lane are two 16-bit words of the 64-byte record.
// The two halves of a warp work independently (shuffles carry a 16-lane
// mask), so a half-warp is the unit of work in every kernel.
//
// All arithmetic is fp32.  Softmax runs in the log2 domain (logits scaled by
// log2(e)/sqrt(128), exp2).

#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <algorithm>
#include <mutex>
#include <type_traits>
#include <string>
#include <vector>

#include "hsq_internal.h"

namespace {

using hsq::kDim;

constexpr float kRsqrtD = 0.08838834764831845f;                 // 1/sqrt(128)
constexpr float kLogitScaleLog2 = 0.12751743074960003f;         // log2(e)/sqrt(128)
constexpr int kThreads = 256;                                   // all kernels but encode
constexpr int kHalves = kThreads / 16;
constexpr int kRouteGroupsPerCta = 128;
constexpr int kFetchBatchBytes = 17408;                          // fetched records staged per pass
constexpr int kMaxFetchChunksPerThread = (kFetchBatchBytes / 16 + kThreads - 1) / kThreads;

// ---------------------------------------------------------------------------
// Parameter blocks (passed by value).
// ---------------------------------------------------------------------------

struct Tables {
    const float* cb;        // c4[16] | t4[15] pad | c3[8] | t3[7] pad
    const float* rope_hi;   // [n_hi][cos 64 | sin 64]
    const float* rope_lo;   // [256][cos 64 | sin 64]
    int max_pos;
};

struct CacheView {
    int B, T, G, N, Hkv, Hq, beta, max_l1, W;
    const uint8_t* l1_kc; const uint8_t* l1_vc; const float* l1_kn; const float* l1_vn;
    const int32_t* l1_pos; const int32_t* l1_count;
    const uint8_t* l2_kc; const uint8_t* l2_vc; const float* l2_kn; const float* l2_vn;
    const uint8_t* l2_cnt;
    const uint8_t* l3;
    const uint32_t* l1_bitmap;
    const int8_t* signs;
    const uint8_t* staging;
};

// ---------------------------------------------------------------------------
// Half-warp helpers.
// ---------------------------------------------------------------------------

__device__ __forceinline__ unsigned half_mask() { return 0xFFFFu << (threadIdx.x & 16); }
__device__ __forceinline__ int hlane() { return threadIdx.x & 15; }

__device__ __forceinline__ float half_sum(float v, unsigned m) {
    v += __shfl_xor_sync(m, v, 1, 16);
    v += __shfl_xor_sync(m, v, 2, 16);
    v += __shfl_xor_sync(m, v, 4, 16);
    v += __shfl_xor_sync(m, v, 8, 16);
    return v;
}

// Unnormalised Sylvester-Hadamard transform of the half-warp's 128-vector.
__device__ __forceinline__ void fwht(float v[8], unsigned m) {
#pragma unroll
    for (int i = 0; i < 8; i += 2) {  // index bit 0
        float a = v[i], b = v[i + 1];
        v[i] = a + b; v[i + 1] = a - b;
    }
#pragma unroll
    for (int base = 0; base < 8; base += 4) {  // index bit 1
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            float a = v[base + k], b = v[base + k + 2];
            v[base + k] = a + b; v[base + k + 2] = a - b;
        }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {  // index bit 6
        float a = v[k], b = v[k + 4];
        v[k] = a + b; v[k + 4] = a - b;
    }
    const int l = hlane();
#pragma unroll
    for (int s = 1; s < 16; s <<= 1) {  // index bits 2..5 = lane bits 0..3
        const float sgn = (l & s) ? -1.f : 1.f;  // upper lane: p - v, lower lane: v + p
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float p = __shfl_xor_sync(m, v[i], s, 16);
            v[i] = fmaf(sgn, v[i], p);
        }
    }
}

__device__ __forceinline__ void load_signs(float s[8], const float* s_sign) {
    const int l = hlane();
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        s[k] = s_sign[4 * l + k];
        s[4 + k] = s_sign[64 + 4 * l + k];
    }
}

// RoPE at position p by angle addition: p = 256 a + c.
__device__ __forceinline__ void rope(float v[8], int p, const Tables& tb) {
    const int l = hlane();
    const float* rh = tb.rope_hi + (size_t)(p >> 8) * kDim;
    const float* rl = tb.rope_lo + (size_t)(p & 255) * kDim;
    const float4 ch = __ldg(reinterpret_cast<const float4*>(rh + 4 * l));
    const float4 sh = __ldg(reinterpret_cast<const float4*>(rh + 64 + 4 * l));
    const float4 cl = __ldg(reinterpret_cast<const float4*>(rl + 4 * l));
    const float4 sl = __ldg(reinterpret_cast<const float4*>(rl + 64 + 4 * l));
    const float cA[4] = {ch.x, ch.y, ch.z, ch.w}, sA[4] = {sh.x, sh.y, sh.z, sh.w};
    const float cB[4] = {cl.x, cl.y, cl.z, cl.w}, sB[4] = {sl.x, sl.y, sl.z, sl.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float c = fmaf(cA[k], cB[k], -sA[k] * sB[k]);
        const float s = fmaf(sA[k], cB[k], cA[k] * sB[k]);
        const float lo = v[k], hi = v[4 + k];
        v[k] = fmaf(lo, c, -hi * s);
        v[4 + k] = fmaf(hi, c, lo * s);
    }
}

__device__ __forceinline__ int quant4(float y, const float* t) {
    int c = (y > t[7]) ? 8 : 0;
    c += (y > t[c + 3]) ? 4 : 0;
    c += (y > t[c + 1]) ? 2 : 0;
    c += (y > t[c]) ? 1 : 0;
    return c;
}

__device__ __forceinline__ int quant3(float y, const float* t) {
    int c = (y > t[3]) ? 4 : 0;
    c += (y > t[c + 1]) ? 2 : 0;
    c += (y > t[c]) ? 1 : 0;
    return c;
}

// TurboQuant forward: y = Pi (x / n) with Pi = H diag(s) / sqrt(d).  Returns n.
__device__ __forceinline__ float tq_rotate(float x[8], float y[8], const float sg[8], unsigned m) {
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) ss = fmaf(x[i], x[i], ss);
    ss = half_sum(ss, m);
    const float n = sqrtf(ss);
    const float inv = n > 0.f ? 1.0f / n : 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) y[i] = x[i] * inv * sg[i];
    fwht(y, m);
#pragma unroll
    for (int i = 0; i < 8; ++i) y[i] *= kRsqrtD;
    return n;
}

// 4-bit codes of the lane's 8 coordinates as the two 16-bit words of the record.
__device__ __forceinline__ void pack4(const float y[8], const float* t4, uint16_t& lo, uint16_t& hi) {
    uint32_t a = 0, b = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        a |= (uint32_t)quant4(y[k], t4) << (4 * k);
        b |= (uint32_t)quant4(y[4 + k], t4) << (4 * k);
    }
    lo = (uint16_t)a;
    hi = (uint16_t)b;
}

__device__ __forceinline__ void unpack4(uint32_t lo, uint32_t hi, const float* c4, float scale, float v[8]) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        v[k] = c4[(lo >> (4 * k)) & 15] * scale;
        v[4 + k] = c4[(hi >> (4 * k)) & 15] * scale;
    }
}

// 3-bit record (12 words): the lane's fields start at bits 12 l and 192 + 12 l.
__device__ __forceinline__ void unpack3(const uint32_t* __restrict__ rec, const float* c3, float scale, float v[8]) {
    const int l = hlane();
    const int bit = 12 * l, w = bit >> 5, sh = bit & 31;
    const int w1 = min(w + 1, 5);
    const uint32_t a0 = __ldg(rec + w), a1 = __ldg(rec + w1);
    const uint32_t b0 = __ldg(rec + 6 + w), b1 = __ldg(rec + 6 + w1);
    const uint32_t fa = __funnelshift_r(a0, a1, sh) & 0xFFFu;
    const uint32_t fb = __funnelshift_r(b0, b1, sh) & 0xFFFu;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        v[k] = c3[(fa >> (3 * k)) & 7] * scale;
        v[4 + k] = c3[(fb >> (3 * k)) & 7] * scale;
    }
}

__device__ __forceinline__ void load_f32x8(const float* __restrict__ p, float v[8]) {
    const int l = hlane();
    const float4 a = __ldg(reinterpret_cast<const float4*>(p + 4 * l));
    const float4 b = __ldg(reinterpret_cast<const float4*>(p + 64 + 4 * l));
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

__device__ __forceinline__ void load_bf16x8(const uint16_t* __restrict__ p, float v[8]) {
    const int l = hlane();
    const uint2 a = __ldg(reinterpret_cast<const uint2*>(p + 4 * l));
    const uint2 b = __ldg(reinterpret_cast<const uint2*>(p + 64 + 4 * l));
    v[0] = __uint_as_float(a.x << 16); v[1] = __uint_as_float(a.x & 0xFFFF0000u);
    v[2] = __uint_as_float(a.y << 16); v[3] = __uint_as_float(a.y & 0xFFFF0000u);
    v[4] = __uint_as_float(b.x << 16); v[5] = __uint_as_float(b.x & 0xFFFF0000u);
    v[6] = __uint_as_float(b.y << 16); v[7] = __uint_as_float(b.y & 0xFFFF0000u);
}

__device__ __forceinline__ void load_f32x8_smem(const float* p, float v[8]) {
    const int l = hlane();
    const float4 a = *reinterpret_cast<const float4*>(p + 4 * l);
    const float4 b = *reinterpret_cast<const float4*>(p + 64 + 4 * l);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

__device__ __forceinline__ void store_f32x8(float* __restrict__ p, const float v[8]) {
    const int l = hlane();
    *reinterpret_cast<float4*>(p + 4 * l) = make_float4(v[0], v[1], v[2], v[3]);
    *reinterpret_cast<float4*>(p + 64 + 4 * l) = make_float4(v[4], v[5], v[6], v[7]);
}

__device__ __forceinline__ void load_tables(float* s_cb, float* s_sign, const Tables& tb,
                                            const int8_t* __restrict__ signs) {
    for (int i = threadIdx.x; i < hsq::kCodebookFloats; i += blockDim.x) s_cb[i] = tb.cb[i];
    for (int i = threadIdx.x; i < kDim; i += blockDim.x) s_sign[i] = (float)signs[i];
}

__device__ __forceinline__ int checked_pos(int p, const Tables& tb, int* err) {
    if (p < 0 || p >= tb.max_pos) {
        atomicOr(err, HSQ_DEVERR_POS);
        p = p < 0 ? 0 : tb.max_pos - 1;
    }
    return p;
}

__device__ __forceinline__ bool in_l1(const CacheView& c, int b, int t) {
    const uint32_t w = __ldg(c.l1_bitmap + (size_t)b * c.W + (t >> 5));
    return (w >> (t & 31)) & 1u;
}

// Block-wide exclusive scan of one int per thread (blockDim.x <= 1024).
__device__ int block_exclusive_scan(int v, int* s_warp, int& total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int t = lane < nw ? s_warp[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t += y;
        }
        if (lane < nw) s_warp[lane] = t;
    }
    __syncthreads();
    total = s_warp[nw - 1];
    const int before = warp > 0 ? s_warp[warp - 1] : 0;
    __syncthreads();
    return before + x - v;
}

// ---------------------------------------------------------------------------
// Encode, stage 1: L1 slot prefix per bitmap word, L1 position list, counts.
// One CTA per sequence.
// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(1024) l1_index_kernel(CacheView c, int32_t* __restrict__ l1_pos,
                                                        int32_t* __restrict__ l1_count,
                                                        int32_t* __restrict__ prefix, int* err) {
    __shared__ int s_warp[32];
    const int b = blockIdx.x;
    const int W = c.W;
    const int per = (W + blockDim.x - 1) / blockDim.x;
    const int w0 = min(W, (int)threadIdx.x * per), w1 = min(W, w0 + per);
    auto word = [&](int w) -> uint32_t {
        uint32_t x = c.l1_bitmap[(size_t)b * W + w];
        const int valid = c.T - 32 * w;
        if (valid < 32) x &= (1u << valid) - 1u;
        return x;
    };
    int local = 0;
    for (int w = w0; w < w1; ++w) local += __popc(word(w));
    int total;
    int run = block_exclusive_scan(local, s_warp, total);
    for (int w = w0; w < w1; ++w) {
        uint32_t x = word(w);
        prefix[(size_t)b * W + w] = run;
        while (x) {
            const int bit = __ffs(x) - 1;
            x &= x - 1;
            if (run < c.max_l1) l1_pos[(size_t)b * c.max_l1 + run] = 32 * w + bit;
            ++run;
        }
    }
    if (threadIdx.x == 0) {
        l1_count[b] = min(total, c.max_l1);
        if (total > c.max_l1) atomicOr(err, HSQ_DEVERR_L1_OVER);
    }
}

// ---------------------------------------------------------------------------
// Encode, stage 2: one CTA per (group g, KV head h, sequence b), one warp per
// token: half 0 encodes the key, half 1 the value.
// ---------------------------------------------------------------------------

struct EncodeOut {
    uint8_t* l1_kc; uint8_t* l1_vc; float* l1_kn; float* l1_vn;
    uint8_t* l2_kc; uint8_t* l2_vc; float* l2_kn; float* l2_vn; uint8_t* l2_cnt;
    uint8_t* l3;
    const int32_t* prefix;
};

template <int N, bool kBF16>
__global__ void __launch_bounds__(N * 32) encode_kernel(CacheView c, EncodeOut o, const void* __restrict__ Kp,
                                                        const void* __restrict__ Vp, Tables tb) {
    __shared__ float s_cb[hsq::kCodebookFloats];
    __shared__ float s_sign[kDim];
    __shared__ __align__(16) uint8_t s_rec[N * 136];
    __shared__ __align__(16) float s_sum[N][2][kDim];
    __shared__ int s_member[N];
    __shared__ uint32_t s_l2[2][12];

    const int g = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, half = (threadIdx.x >> 4) & 1, l = hlane();
    const unsigned m = half_mask();
    load_tables(s_cb, s_sign, tb, c.signs);
    if (threadIdx.x < 24) (&s_l2[0][0])[threadIdx.x] = 0u;
    __syncthreads();
    const float* t4 = s_cb + 16;
    const float* t3 = s_cb + 40;
    float sg[8];
    load_signs(sg, s_sign);

    const int t = g * N + warp;
    const bool in_ctx = t < c.T;
    bool is_l1 = false;
    int slot = 0;
    if (in_ctx) {
        const uint32_t w = __ldg(c.l1_bitmap + (size_t)b * c.W + (t >> 5));
        is_l1 = (w >> (t & 31)) & 1u;
        if (is_l1) slot = o.prefix[(size_t)b * c.W + (t >> 5)] + __popc(w & ((1u << (t & 31)) - 1u));
    }

    float x[8];
    if (in_ctx) {
        const size_t off = (((size_t)b * c.Hkv + h) * c.T + t) * kDim;
        if (kBF16) load_bf16x8(static_cast<const uint16_t*>(half ? Vp : Kp) + off, x);
        else load_f32x8(static_cast<const float*>(half ? Vp : Kp) + off, x);
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] = 0.f;
    }

    // L3: TQ4 of the raw (pre-RoPE) key / value
    float y[8];
    const float n = tq_rotate(x, y, sg, m);
    uint16_t lo, hi;
    pack4(y, t4, lo, hi);
    {
        uint8_t* row = s_rec + (half ? N * 64 : 0) + warp * 64;
        reinterpret_cast<uint16_t*>(row)[l] = lo;
        reinterpret_cast<uint16_t*>(row + 32)[l] = hi;
        if (l == 0) reinterpret_cast<float*>(s_rec + N * 128)[half * N + warp] = n;
    }

    // RoPE'd key (half 0) for L1 and for the group summary; values as they are
    float xr[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) xr[i] = x[i];
    if (half == 0 && in_ctx) rope(xr, t, tb);

    if (is_l1 && slot < c.max_l1) {
        const size_t so = ((size_t)b * c.Hkv + h) * c.max_l1 + slot;
        if (half == 0) {
            float yr[8];
            tq_rotate(xr, yr, sg, m);  // same norm as the raw key (RoPE is norm preserving)
            uint16_t klo, khi;
            pack4(yr, t4, klo, khi);
            reinterpret_cast<uint16_t*>(o.l1_kc + so * 64)[l] = klo;
            reinterpret_cast<uint16_t*>(o.l1_kc + so * 64 + 32)[l] = khi;
            if (l == 0) o.l1_kn[so] = n;
        } else {
            reinterpret_cast<uint16_t*>(o.l1_vc + so * 64)[l] = lo;
            reinterpret_cast<uint16_t*>(o.l1_vc + so * 64 + 32)[l] = hi;
            if (l == 0) o.l1_vn[so] = n;
        }
    }

    const bool member = in_ctx && !is_l1;
    if (member) {
        float* row = &s_sum[warp][half][0];
        *reinterpret_cast<float4*>(row + 4 * l) = make_float4(xr[0], xr[1], xr[2], xr[3]);
        *reinterpret_cast<float4*>(row + 64 + 4 * l) = make_float4(xr[4], xr[5], xr[6], xr[7]);
    }
    if (threadIdx.x == warp * 32) s_member[warp] = member ? 1 : 0;
    __syncthreads();

    // L3 record out (16-byte chunks; through the host link when L3 is pinned host memory)
    {
        uint4* dst = reinterpret_cast<uint4*>(o.l3 + (((size_t)b * c.Hkv + h) * c.G + g) * (N * 136));
        const uint4* src = reinterpret_cast<const uint4*>(s_rec);
        for (int i = threadIdx.x; i < N * 136 / 16; i += blockDim.x) dst[i] = src[i];
    }

    // L2 summary: mean over members in token order, then TQ3
    if (warp == 0) {
        int cnt = 0;
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.f;
        for (int k = 0; k < N; ++k) {
            if (!s_member[k]) continue;
            ++cnt;
            const float* row = &s_sum[k][half][0];
            const float4 a = *reinterpret_cast<const float4*>(row + 4 * l);
            const float4 bq = *reinterpret_cast<const float4*>(row + 64 + 4 * l);
            acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
            acc[4] += bq.x; acc[5] += bq.y; acc[6] += bq.z; acc[7] += bq.w;
        }
        if (cnt > 0) {
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = acc[i] / (float)cnt;
        }
        float ys[8];
        const float ns = tq_rotate(acc, ys, sg, m);
        uint32_t fa = 0, fb = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            fa |= (uint32_t)quant3(ys[k], t3) << (3 * k);
            fb |= (uint32_t)quant3(ys[4 + k], t3) << (3 * k);
        }
        uint32_t* w = s_l2[half];
        const int bit = 12 * l, wi = bit >> 5, sh = bit & 31;
        atomicOr(&w[wi], fa << sh);
        if (sh > 20) atomicOr(&w[wi + 1], fa >> (32 - sh));
        atomicOr(&w[6 + wi], fb << sh);
        if (sh > 20) atomicOr(&w[6 + wi + 1], fb >> (32 - sh));
        __syncwarp();
        const size_t go = ((size_t)b * c.Hkv + h) * c.G + g;
        uint32_t* dst = reinterpret_cast<uint32_t*>((half ? o.l2_vc : o.l2_kc) + go * 48);
        if (l < 12) dst[l] = w[l];
        if (l == 0) (half ? o.l2_vn : o.l2_kn)[go] = ns;
        if (threadIdx.x == 0 && h == 0) o.l2_cnt[(size_t)b * c.G + g] = (uint8_t)cnt;
    }
}

// ---------------------------------------------------------------------------
// Asynchronous global -> shared staging of device-resident inputs.
// ---------------------------------------------------------------------------

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    const unsigned s = (unsigned)__cvta_generic_to_shared(dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
    const unsigned s = (unsigned)__cvta_generic_to_shared(dst);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(s), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }

// bytes: a multiple of 16, both addresses 16-byte aligned
__device__ __forceinline__ void stage16(void* dst, const void* src, int bytes) {
    uint8_t* d = static_cast<uint8_t*>(dst);
    const uint8_t* s = static_cast<const uint8_t*>(src);
    for (int i = threadIdx.x * 16; i < bytes; i += blockDim.x * 16) cp_async16(d + i, s + i);
}

__device__ __forceinline__ void stage4(float* dst, const float* src, int n) {
    for (int i = threadIdx.x; i < n; i += blockDim.x) cp_async4(dst + i, src + i);
}

// signs of the lane's 8 dims straight from global memory
__device__ __forceinline__ void load_signs_global(float s[8], const int8_t* __restrict__ signs) {
    const int l = hlane();
    const char4 a = *reinterpret_cast<const char4*>(signs + 4 * l);
    const char4 b = *reinterpret_cast<const char4*>(signs + 64 + 4 * l);
    s[0] = a.x; s[1] = a.y; s[2] = a.z; s[3] = a.w;
    s[4] = b.x; s[5] = b.y; s[6] = b.z; s[7] = b.w;
}

// 3-bit record held in shared memory
__device__ __forceinline__ void unpack3_smem(const uint8_t* rec8, const float* c3, float scale, float v[8]) {
    const uint32_t* rec = reinterpret_cast<const uint32_t*>(rec8);
    const int l = hlane();
    const int bit = 12 * l, w = bit >> 5, sh = bit & 31;
    const int w1 = min(w + 1, 5);
    const uint32_t fa = __funnelshift_r(rec[w], rec[w1], sh) & 0xFFFu;
    const uint32_t fb = __funnelshift_r(rec[6 + w], rec[6 + w1], sh) & 0xFFFu;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        v[k] = c3[(fa >> (3 * k)) & 7] * scale;
        v[4 + k] = c3[(fb >> (3 * k)) & 7] * scale;
    }
}

// ---------------------------------------------------------------------------
// Top-beta selection by radix select over order-preserving score keys.
// ---------------------------------------------------------------------------

struct RouteArgs {
    const float* q; const int32_t* pos; int32_t* sel; float* scores; int* counters; int* err;
};

__device__ __forceinline__ uint32_t ordered_key(float s) {
    if (s == -INFINITY) return 0u;
    const uint32_t u = __float_as_uint(s);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_to_float(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

constexpr int kSelBins = 2048;          // histogram bins of the bucket select (8 per thread)
constexpr int kSelMaxGroups = 32768;
constexpr int kSelCand = 32;            // boundary candidates ranked in one warp

struct __align__(16) SelectSmem {
    int hist[kSelBins];
    uint32_t taken[kSelMaxGroups / 32];
    uint32_t cand_key[kSelCand];
    int cand_g[kSelCand];
    uint32_t red[3][8];
    int warp[32];
    int bstar, above, bcnt, ncand;
};

// Top-beta selection by the whole block (256 threads).  s_keys[0..G) are
// order-preserving keys of the fp32 group scores (0 = empty group, never
// selected).  The beta largest keys (ties to the lower group) go, in ascending
// group order and -1 padded, to sel_row (global) and, when s_out is not null,
// to s_out (shared).
//
// Bucket select: the keys still in play, [lo, hi], are histogrammed (first
// pass: kSelBins equal-width bins of the fp32 score; later passes: power-of-
// two-wide bins of the key), a blocked scan from the top finds the bin that
// holds the beta-th key, every key of a higher bin is taken, and the
// boundary bin's keys are ranked exactly (key, then group index) when there
// are at most 32 of them; otherwise [lo, hi] shrinks to that bin and the
// pass repeats.  If all keys left are equal, the lowest groups are taken.
// Both bin functions are monotone in the key, so a bin is a contiguous key
// range and the result is exact.
__device__ void select_top_beta(const uint32_t* s_keys, int G, int beta, int32_t* __restrict__ sel_row,
                                int* s_out, SelectSmem& ss) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nt = blockDim.x;
    const unsigned full = 0xffffffffu;

    // count, max and min of the non-empty keys (every thread reduces the per-warp values itself)
    int ne;
    uint32_t lo = 0xFFFFFFFFu, hi = 0u;
    {
        int c = 0;
        uint32_t mx = 0u, mn = 0xFFFFFFFFu;
        for (int g = tid; g < G; g += nt) {
            const uint32_t v = s_keys[g];
            if (v != 0u) { ++c; mx = max(mx, v); mn = min(mn, v); }
        }
        c = __reduce_add_sync(full, c);
        mx = __reduce_max_sync(full, mx);
        mn = __reduce_min_sync(full, mn);
        if (lane == 0) { ss.red[0][warp] = (uint32_t)c; ss.red[1][warp] = mx; ss.red[2][warp] = mn; }
        for (int g = tid; g < (G + 31) / 32; g += nt) ss.taken[g] = 0u;
        __syncthreads();
        ne = 0;
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) {
            ne += (int)ss.red[0][w];
            hi = max(hi, ss.red[1][w]);
            lo = min(lo, ss.red[2][w]);
        }
    }

    // mode 0: take every non-empty group; 1: keys > bhi plus the ranked
    // boundary candidates; 2: keys > kstar plus the first `need` equal to kstar
    int mode = 0, above = 0, need = 0;
    uint32_t bhi = 0u, kstar = 0u;
    if (ne > beta) {
        const float smin = key_to_float(lo), smax = key_to_float(hi);
        const float fscale = (float)kSelBins / (smax - smin);
        const bool float_ok = isfinite(fscale) && smax > smin;
        for (int level = 0; level < 8; ++level) {
            if (lo == hi) { mode = 2; kstar = lo; need = beta - above; break; }
            const bool fl = level == 0 && float_ok;
            const uint32_t span = hi - lo;
            const int bits = 32 - __clz(span);
            const int shift = bits > 11 ? bits - 11 : 0;
            auto bin_of = [&](uint32_t v) -> int {
                if (fl) return min(max((int)((key_to_float(v) - smin) * fscale), 0), kSelBins - 1);
                return (int)((v - lo) >> shift);
            };
            for (int i = tid; i < kSelBins; i += nt) ss.hist[i] = 0;
            __syncthreads();
            for (int g = tid; g < G; g += nt) {
                const uint32_t v = s_keys[g];
                if (v != 0u && v >= lo && v <= hi) atomicAdd(&ss.hist[bin_of(v)], 1);
            }
            __syncthreads();
            // blocked scan from the top: thread t owns bins [B - 8(t+1), B - 8t)
            const int top = kSelBins - 8 * tid;
            const int4 h0 = *reinterpret_cast<const int4*>(&ss.hist[top - 8]);
            const int4 h1 = *reinterpret_cast<const int4*>(&ss.hist[top - 4]);
            const int hv[8] = {h1.w, h1.z, h1.y, h1.x, h0.w, h0.z, h0.y, h0.x};  // descending bins
            int local = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) local += hv[i];
            int tot;
            int run = above + block_exclusive_scan(local, ss.warp, tot);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (run < beta && run + hv[i] >= beta) { ss.bstar = top - 1 - i; ss.above = run; ss.bcnt = hv[i]; }
                run += hv[i];
            }
            if (tid == 0) ss.ncand = 0;
            __syncthreads();
            const int bstar = ss.bstar, bcnt = ss.bcnt;
            above = ss.above;
            need = beta - above;
            // the boundary bin's members: gather (when few) and their exact key range
            uint32_t bmx = 0u, bmn = 0xFFFFFFFFu;
            for (int g = tid; g < G; g += nt) {
                const uint32_t v = s_keys[g];
                if (v != 0u && v >= lo && v <= hi && bin_of(v) == bstar) {
                    bmx = max(bmx, v);
                    bmn = min(bmn, v);
                    if (bcnt <= kSelCand) {
                        const int slot = atomicAdd(&ss.ncand, 1);
                        ss.cand_key[slot] = v;
                        ss.cand_g[slot] = g;
                    }
                }
            }
            bmx = __reduce_max_sync(full, bmx);
            bmn = __reduce_min_sync(full, bmn);
            if (lane == 0) { ss.red[1][warp] = bmx; ss.red[2][warp] = bmn; }
            __syncthreads();
            uint32_t blo_b = 0xFFFFFFFFu, bhi_b = 0u;
#pragma unroll
            for (int w = 0; w < kThreads / 32; ++w) {
                bhi_b = max(bhi_b, ss.red[1][w]);
                blo_b = min(blo_b, ss.red[2][w]);
            }
            if (bcnt <= kSelCand) {
                if (warp == 0) {
                    const uint32_t ck = lane < bcnt ? ss.cand_key[lane] : 0u;
                    const int cg = lane < bcnt ? ss.cand_g[lane] : -1;
                    int rank = 0;
                    for (int j = 0; j < bcnt; ++j) {
                        const uint32_t kj = __shfl_sync(full, ck, j);
                        const int gj = __shfl_sync(full, cg, j);
                        rank += (kj > ck) || (kj == ck && gj < cg);
                    }
                    if (lane < bcnt && rank < need) atomicOr(&ss.taken[cg >> 5], 1u << (cg & 31));
                }
                mode = 1;
                bhi = bhi_b;
                __syncthreads();
                break;
            }
            lo = blo_b;  // crowded boundary bin: continue inside it
            hi = bhi_b;
            __syncthreads();
        }
    }

    // ordered placement: thread t owns the contiguous groups [per*t, per*t + per)
    const int per = (G + nt - 1) / nt;
    const int i0 = min(G, tid * per), i1 = min(G, i0 + per);
    auto take_of = [&](int g, uint32_t v, int eq_rank) -> bool {
        if (mode == 0) return v != 0u;
        if (mode == 1) return v > bhi || (v != 0u && ((ss.taken[g >> 5] >> (g & 31)) & 1u));
        return v > kstar || (v == kstar && eq_rank < need);
    };
    int nsel = 0, neq = 0;
    for (int g = i0; g < i1; ++g) {
        const uint32_t v = s_keys[g];
        if (mode == 2) { nsel += (v > kstar); neq += (v == kstar); }
        else nsel += take_of(g, v, 0);
    }
    int total;
    const int packed = block_exclusive_scan(nsel | (neq << 16), ss.warp, total);
    int pos_gt = packed & 0xFFFF, eq_before = packed >> 16;
    for (int g = i0; g < i1; ++g) {
        const uint32_t v = s_keys[g];
        const bool take = take_of(g, v, eq_before);
        const int pos = mode == 2 ? pos_gt + min(eq_before, need) : pos_gt;
        if (take && pos < beta) {
            sel_row[pos] = g;
            if (s_out) s_out[pos] = g;
        }
        if (mode == 2) { pos_gt += (v > kstar); eq_before += (v == kstar); }
        else pos_gt += take;
    }
    const int n_sel = mode == 0 ? ne : beta;
    for (int i = n_sel + tid; i < beta; i += nt) {
        sel_row[i] = -1;
        if (s_out) s_out[i] = -1;
    }
}

// ---------------------------------------------------------------------------
// Route (standalone call): grid = (ceil(G / 128), B * Hkv).  Each CTA stages
// its 128 groups' summary keys in shared memory, scores them against the
// aggregated rotated query, and the last CTA of a (b, h) selects.
// ---------------------------------------------------------------------------

__host__ __device__ inline unsigned al16(size_t x) { return (unsigned)((x + 15) & ~(size_t)15); }

__host__ __device__ inline unsigned route_smem_bytes(int G) {
    return al16((size_t)G * 4) + kRouteGroupsPerCta * (48 + 4 + 1);
}

template <int R>
__global__ void __launch_bounds__(kThreads) route_kernel(CacheView c, RouteArgs a, Tables tb) {
    extern __shared__ __align__(16) uint8_t s_dyn[];
    __shared__ __align__(16) float s_cb[hsq::kCodebookFloats];
    __shared__ __align__(16) float s_q[R][kDim];
    __shared__ SelectSmem s_ss;
    __shared__ int s_flag;

    const int bh = blockIdx.y, b = bh / c.Hkv, h = bh % c.Hkv;
    const int tid = threadIdx.x, hw = tid >> 4, l = hlane();
    const unsigned m = half_mask();
    uint32_t* s_keys = reinterpret_cast<uint32_t*>(s_dyn);
    uint8_t* s_codes = s_dyn + al16((size_t)c.G * 4);
    float* s_kn = reinterpret_cast<float*>(s_codes + kRouteGroupsPerCta * 48);
    uint8_t* s_cnt = reinterpret_cast<uint8_t*>(s_kn + kRouteGroupsPerCta);

    const int g_begin = blockIdx.x * kRouteGroupsPerCta;
    const int ng = min(c.G, g_begin + kRouteGroupsPerCta) - g_begin;
    stage16(s_codes, c.l2_kc + ((size_t)bh * c.G + g_begin) * 48, ng * 48);
    stage4(s_kn, c.l2_kn + (size_t)bh * c.G + g_begin, ng);
    if (tid < hsq::kCodebookFloats / 4) cp_async16(s_cb + 4 * tid, tb.cb + 4 * tid);
    for (int i = tid; i < ng; i += kThreads) s_cnt[i] = __ldg(c.l2_cnt + (size_t)b * c.G + g_begin + i);
    float sg[8];
    load_signs_global(sg, c.signs);

    // rotated, RoPE'd query of each query head of this KV head
    if (hw < R) {
        const int j = h * R + hw;
        const int p = checked_pos(__ldg(a.pos + b), tb, a.err);
        float x[8];
        load_f32x8(a.q + ((size_t)b * c.Hq + j) * kDim, x);
        rope(x, p, tb);
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] *= sg[i];
        fwht(x, m);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            s_q[hw][4 * l + k] = x[k] * kRsqrtD;
            s_q[hw][64 + 4 * l + k] = x[4 + k] * kRsqrtD;
        }
    }
    cp_async_wait_all();
    __syncthreads();
    float gq[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int jj = 0; jj < R; ++jj) {
            s0 += s_q[jj][4 * l + k];
            s1 += s_q[jj][64 + 4 * l + k];
        }
        gq[k] = s0;
        gq[4 + k] = s1;
    }
    const float* c3 = s_cb + 32;
    for (int i = hw; i < ng; i += kHalves) {
        float score = -INFINITY;
        if (s_cnt[i] > 0) {
            float v[8];
            unpack3_smem(s_codes + i * 48, c3, 1.0f, v);
            float d = 0.f;
#pragma unroll
            for (int k = 0; k < 8; ++k) d = fmaf(gq[k], v[k], d);
            d = half_sum(d, m);
            score = s_kn[i] * d;
        }
        if (l == 0) a.scores[(size_t)bh * c.G + g_begin + i] = score;
    }

    __syncthreads();
    if (tid == 0) {
        __threadfence();
        const int ticket = atomicAdd(a.counters + bh, 1);
        s_flag = (ticket == (int)gridDim.x - 1);
        if (s_flag) __threadfence();
    }
    __syncthreads();
    if (!s_flag) return;
    for (int g = tid; g < c.G; g += kThreads) s_keys[g] = ordered_key(__ldcg(a.scores + (size_t)bh * c.G + g));
    __syncthreads();
    select_top_beta(s_keys, c.G, c.beta, a.sel + (size_t)bh * c.beta, nullptr, s_ss);
    if (tid == 0) a.counters[bh] = 0;
}

// ---------------------------------------------------------------------------
// Selection validity: entries must be -1 or in [0, G), non-negative entries
// strictly ascending and before any -1.
// ---------------------------------------------------------------------------

__device__ __forceinline__ int valid_sel(const int32_t* __restrict__ row, int i, int G, int* err) {
    const int g = __ldg(row + i);
    if (g < 0) return -1;
    bool ok = g < G;
    if (i > 0) {
        const int p = __ldg(row + i - 1);
        ok = ok && p >= 0 && p < g;
    }
    if (!ok) {
        atomicOr(err, HSQ_DEVERR_SEL);
        return -1;
    }
    return g;
}

// ---------------------------------------------------------------------------
// Fetch + dequantise (standalone): one CTA per (selected slot i, b*Hkv + h).
// ---------------------------------------------------------------------------

struct FetchArgs {
    const int32_t* sel; float* k_out; float* v_out; uint8_t* valid; uint8_t* staging; int* err;
};

template <int N>
__global__ void __launch_bounds__(kThreads) fetch_kernel(CacheView c, FetchArgs a, Tables tb) {
    __shared__ float s_cb[hsq::kCodebookFloats];
    __shared__ float s_sign[kDim];
    __shared__ __align__(16) uint8_t s_rec[N * 136];
    __shared__ int s_g;

    const int i = blockIdx.x, bh = blockIdx.y, b = bh / c.Hkv;
    const int hw = threadIdx.x >> 4, l = hlane();
    const unsigned m = half_mask();
    load_tables(s_cb, s_sign, tb, c.signs);
    if (threadIdx.x == 0) s_g = valid_sel(a.sel + (size_t)bh * c.beta, i, c.G, a.err);
    __syncthreads();
    const int g = s_g;
    constexpr int kChunks = N * 136 / 16;
    uint4* srec = reinterpret_cast<uint4*>(s_rec);
    for (int k = threadIdx.x; k < kChunks; k += blockDim.x) {
        uint4 v = make_uint4(0, 0, 0, 0);
        if (g >= 0) v = __ldcg(reinterpret_cast<const uint4*>(c.l3 + ((size_t)bh * c.G + g) * (N * 136)) + k);
        srec[k] = v;
        if (a.staging) reinterpret_cast<uint4*>(a.staging + ((size_t)bh * c.beta + i) * (N * 136))[k] = v;
    }
    __syncthreads();
    if (hw >= N) return;
    float sg[8];
    load_signs(sg, s_sign);
    const int t = g * N + hw;
    const bool have = g >= 0 && t < c.T;
    const size_t oo = (((size_t)bh * c.beta + i) * N + hw) * kDim;
    float kx[8], vx[8];
    if (have) {
        const float* c4 = s_cb;
        const float* norms = reinterpret_cast<const float*>(s_rec + N * 128);
        const uint16_t* kr = reinterpret_cast<const uint16_t*>(s_rec + hw * 64);
        const uint16_t* vr = reinterpret_cast<const uint16_t*>(s_rec + N * 64 + hw * 64);
        unpack4(kr[l], kr[16 + l], c4, 1.0f, kx);
        unpack4(vr[l], vr[16 + l], c4, 1.0f, vx);
        fwht(kx, m);
        fwht(vx, m);
        const float kn = norms[hw] * kRsqrtD, vn = norms[N + hw] * kRsqrtD;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            kx[q] *= sg[q] * kn;
            vx[q] *= sg[q] * vn;
        }
        rope(kx, t, tb);
    } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) kx[q] = vx[q] = 0.f;
    }
    if (a.k_out) store_f32x8(a.k_out + oo, kx);
    if (a.v_out) store_f32x8(a.v_out + oo, vx);
    if (a.valid && l == 0)
        a.valid[((size_t)bh * c.beta + i) * N + hw] = (uint8_t)(have && !in_l1(c, b, t));
}

// ---------------------------------------------------------------------------
// Decode step: one thread-block cluster per (b, KV head).  grid = (S, B*Hkv),
// cluster = (S, 1, 1), 256 threads per CTA.  Split s owns a contiguous share
// of the L2 groups and of the L1 slots of its (b, h) and an even share of the
// selected records.  The splits of a (b, h) exchange what they must through
// distributed shared memory and cluster barriers; nothing goes through
// global scratch.
//   1. stage the split's L2 summaries, L1 tokens, the sequence's L1 bitmap,
//      the codebook and the RoPE angle rows it may need (cp.async);
//   2. rotate the query heads; per-head logits of the split's L2 groups and,
//      with kRoute, the routing score n_g * (sum_j q~_j) . c3[codes] (the
//      arithmetic of the routing kernel, so both select the same groups);
//   3. kRoute: distributed top-beta over the splits' scores (cluster_select);
//      otherwise the caller's selection is validated and used;
//   4. gather this split's share of the selected L3 records (zero copy when
//      L3 is host memory) and, while they travel, add the L1 tokens and the
//      unselected non-empty summaries;
//   5. recovered tokens: dequantise, inverse WHT, RoPE at the token's
//      position (per-record base angle plus a small offset), logits against
//      the RoPE'd queries, values kept in the rotated frame;
//   6. the CTA's softmax partial per query head is published; query head j is
//      merged by split j mod S, rotated back to the original frame, stored.
// Each half-warp runs its own online softmax over its entries.
//
// Inputs that do not fit in shared memory (very long contexts) are read in
// place from global memory instead of being staged (the flags below).
// ---------------------------------------------------------------------------

constexpr int kMaxSplits = 16;   // largest (non-portable) cluster
enum : int { kStageL2 = 1, kKeepLogits = 2, kStageL1 = 4, kStageBitmap = 8 };

struct DecodeArgs {
    const float* q; const int32_t* pos; int32_t* sel; float* out; int* err; int from_staging; int flags;
};

struct DecodeLayout {
    int span, l1span, nlev, nb0;
    unsigned l2k, l2v, l2kn, l2vn, cnt, l1k, l1v, l1kn, l1vn, logit, keys, sel, mask, bitmap;
    unsigned lev, b0, off, base, rbits, rec, total;
};

// 4-bit digits of p >> 8 for cache positions p < T
__host__ __device__ inline int rope_levels(int T) {
    int hi = (T - 1) >> 8, n = 0;
    while (hi > 0) {
        ++n;
        hi >>= 4;
    }
    return n;
}

template <int R, int N>
__host__ __device__ inline DecodeLayout decode_layout(int G, int T, int S, int max_l1, int beta, bool route,
                                                      int flags) {
    DecodeLayout L;
    L.span = (G + S - 1) / S;
    L.l1span = (max_l1 + S - 1) / S;
    L.nlev = rope_levels(T);
    L.nb0 = 256 / N;
    constexpr int kBatchRecs = kFetchBatchBytes / (N * 136);
    const size_t row = (size_t)kDim * 4;
    size_t o = 0;
    L.l2k = L.l2v = L.l2kn = L.l2vn = L.cnt = L.l1k = L.l1v = L.l1kn = L.l1vn = L.logit = L.keys = L.bitmap = 0;
    if (flags & kStageL2) {
        L.l2k = (unsigned)o; o = al16(o + (size_t)L.span * 48);
        L.l2v = (unsigned)o; o = al16(o + (size_t)L.span * 48);
        L.l2kn = (unsigned)o; o = al16(o + (size_t)L.span * 4);
        L.l2vn = (unsigned)o; o = al16(o + (size_t)L.span * 4);
        L.cnt = (unsigned)o; o = al16(o + (size_t)L.span);
    }
    if (flags & kStageL1) {
        L.l1k = (unsigned)o; o = al16(o + (size_t)L.l1span * 64);
        L.l1v = (unsigned)o; o = al16(o + (size_t)L.l1span * 64);
        L.l1kn = (unsigned)o; o = al16(o + (size_t)L.l1span * 4);
        L.l1vn = (unsigned)o; o = al16(o + (size_t)L.l1span * 4);
    }
    if (flags & kKeepLogits) { L.logit = (unsigned)o; o = al16(o + (size_t)L.span * R * 4); }
    if (route) { L.keys = (unsigned)o; o = al16(o + (size_t)L.span * 4); }
    if (flags & kStageBitmap) { L.bitmap = (unsigned)o; o = al16(o + (size_t)((T + 31) / 32) * 4); }
    L.sel = (unsigned)o; o = al16(o + (size_t)beta * 4);
    L.mask = (unsigned)o; o = al16(o + (size_t)((L.span + 31) / 32) * 4);
    L.lev = (unsigned)o; o = al16(o + (size_t)L.nlev * 16 * row);
    L.b0 = (unsigned)o; o = al16(o + (size_t)L.nb0 * row);
    L.off = (unsigned)o; o = al16(o + (size_t)N * row);
    L.base = (unsigned)o; o = al16(o + (size_t)kBatchRecs * row);
    L.rbits = (unsigned)o; o = al16(o + (size_t)kBatchRecs * 4);
    const size_t merge = (size_t)(kThreads / 32) * R * hsq::kPartStride * 4;
    L.rec = (unsigned)o; o = al16(o + (kFetchBatchBytes > merge ? (size_t)kFetchBatchBytes : merge));
    L.total = (unsigned)o;
    return L;
}

// 2^x by the special-function unit (relative error about 2^-22); -inf gives 0
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <int R>
struct Softmax {
    float m[R], l[R], acc[R][8];
    __device__ __forceinline__ void init() {
#pragma unroll
        for (int j = 0; j < R; ++j) {
            m[j] = -INFINITY;
            l[j] = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[j][i] = 0.f;
        }
    }
    // add up to two entries with log2-domain logits xa[j], xb[j] and values va, vb
    __device__ __forceinline__ void add2(const float xa[R], const float va[8], bool oka, const float xb[R],
                                         const float vb[8], bool okb) {
#pragma unroll
        for (int j = 0; j < R; ++j) {
            const float a = oka ? xa[j] : -INFINITY, b = okb ? xb[j] : -INFINITY;
            const float mn = fmaxf(m[j], fmaxf(a, b));
            if (mn > m[j]) {
                const float corr = fast_exp2(m[j] - mn);
                l[j] *= corr;
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[j][i] *= corr;
                m[j] = mn;
            }
            const float pa = oka ? fast_exp2(a - m[j]) : 0.f;
            const float pb = okb ? fast_exp2(b - m[j]) : 0.f;
            l[j] += pa + pb;
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[j][i] = fmaf(pa, va[i], fmaf(pb, vb[i], acc[j][i]));
        }
    }
};

__device__ __forceinline__ float merge_weight(float mi, float M) {
    return mi == -INFINITY ? 0.f : fast_exp2(mi - M);
}

// (c1, s1) <- cos/sin of the sum of the two angles, 4 frequencies
__device__ __forceinline__ void angle_add4(float4& c1, float4& s1, const float4 c2, const float4 s2) {
    const float4 c = make_float4(fmaf(c1.x, c2.x, -s1.x * s2.x), fmaf(c1.y, c2.y, -s1.y * s2.y),
                                 fmaf(c1.z, c2.z, -s1.z * s2.z), fmaf(c1.w, c2.w, -s1.w * s2.w));
    const float4 s = make_float4(fmaf(s1.x, c2.x, c1.x * s2.x), fmaf(s1.y, c2.y, c1.y * s2.y),
                                 fmaf(s1.z, c2.z, c1.z * s2.z), fmaf(s1.w, c2.w, c1.w * s2.w));
    c1 = c;
    s1 = s;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// ---------------------------------------------------------------------------
// Distributed top-beta.  What a split publishes to the others of its cluster,
// and its private scratch.
// ---------------------------------------------------------------------------

struct __align__(16) SelPub {
    int ne, n_cand, n_eq, n_mine;
    uint32_t kmin, kmax, bmin, bmax;
    int hist_coarse[kSelBins / 32];
    int hist[kSelBins];
    uint32_t cand_key[kSelCand];
    int cand_g[kSelCand];
    int mine[HSQ_MAX_BETA];
};

struct SelLocal {
    uint32_t red[3][kThreads / 32];
    int warp[32];
    int g[8];
    int off[kMaxSplits + 1];
};

// Every split holds the keys of its own groups [g0, g0 + n) in s_keys (order-
// preserving keys of the fp32 routing scores, 0 = empty group).  On return,
// in every split, s_sel[0..beta) holds the groups of the beta largest keys
// over the whole cluster (ties to the lower group) in ascending order, -1
// padded, and bit i of s_mark is set iff group g0 + i is selected.  The
// result equals select_top_beta over all keys: the same bins at every level
// (float-linear over the score range first, then power-of-two key bins inside
// the boundary bin), with the histograms summed over the splits.  Every split
// computes the same boundary from the same totals, so all of them take the
// same branches and meet at every cluster barrier.
__device__ void cluster_select(const uint32_t* s_keys, int n, int g0, int beta, int* s_sel, uint32_t* s_mark,
                               SelPub& pub, SelLocal& sl) {
    namespace cgx = cooperative_groups;
    cgx::cluster_group cluster = cgx::this_cluster();
    const int S = (int)cluster.num_blocks(), s = (int)cluster.block_rank();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned full = 0xffffffffu;
    // contiguous groups of this thread, for ordered passes
    const int per = (n + kThreads - 1) / kThreads;
    const int i0 = min(n, tid * per), i1 = min(n, i0 + per);

    // count, max and min of the non-empty keys of the cluster
    {
        int c = 0;
        uint32_t mx = 0u, mn = 0xFFFFFFFFu;
        for (int i = tid; i < n; i += kThreads) {
            const uint32_t v = s_keys[i];
            if (v != 0u) { ++c; mx = max(mx, v); mn = min(mn, v); }
        }
        c = __reduce_add_sync(full, c);
        mx = __reduce_max_sync(full, mx);
        mn = __reduce_min_sync(full, mn);
        if (lane == 0) { sl.red[0][warp] = (uint32_t)c; sl.red[1][warp] = mx; sl.red[2][warp] = mn; }
        __syncthreads();
        if (tid == 0) {
            int t = 0;
            uint32_t hx = 0u, lx = 0xFFFFFFFFu;
#pragma unroll
            for (int w = 0; w < kThreads / 32; ++w) {
                t += (int)sl.red[0][w];
                hx = max(hx, sl.red[1][w]);
                lx = min(lx, sl.red[2][w]);
            }
            pub.ne = t; pub.kmax = hx; pub.kmin = lx;
        }
    }
    cluster.sync();
    if (warp == 0) {
        int t = 0;
        uint32_t hx = 0u, lx = 0xFFFFFFFFu;
        if (lane < S) {
            const SelPub* rp = cluster.map_shared_rank(&pub, lane);
            t = rp->ne; hx = rp->kmax; lx = rp->kmin;
        }
        t = __reduce_add_sync(full, t);
        hx = __reduce_max_sync(full, hx);
        lx = __reduce_min_sync(full, lx);
        if (lane == 0) { sl.g[0] = t; sl.g[1] = (int)hx; sl.g[2] = (int)lx; }
    }
    __syncthreads();
    const int NE = sl.g[0];
    uint32_t hi = (uint32_t)sl.g[1], lo = (uint32_t)sl.g[2];

    auto mark = [&](int i) { atomicOr(&s_mark[i >> 5], 1u << (i & 31)); };

    // mode 0: every non-empty group; 1: boundary bin ranked exactly; 2: all keys left equal
    int mode = 0, above = 0, need = 0;
    uint32_t kstar = 0u;
    if (NE > beta) {
        const float smin = key_to_float(lo), smax = key_to_float(hi);
        const float fscale = (float)kSelBins / (smax - smin);
        const bool float_ok = isfinite(fscale) && smax > smin;
        for (int level = 0; level < 8; ++level) {
            if (lo == hi) { mode = 2; kstar = lo; need = beta - above; break; }
            const bool fl = level == 0 && float_ok;
            const int bits = 32 - __clz(hi - lo);
            const int shift = bits > 11 ? bits - 11 : 0;
            auto bin_of = [&](uint32_t v) -> int {
                if (fl) return min(max((int)((key_to_float(v) - smin) * fscale), 0), kSelBins - 1);
                return (int)((v - lo) >> shift);
            };
            for (int i = tid; i < kSelBins; i += kThreads) pub.hist[i] = 0;
            if (tid < kSelBins / 32) pub.hist_coarse[tid] = 0;
            __syncthreads();
            for (int i = tid; i < n; i += kThreads) {
                const uint32_t v = s_keys[i];
                if (v != 0u && v >= lo && v <= hi) {
                    const int bn = bin_of(v);
                    atomicAdd(&pub.hist[bn], 1);
                    atomicAdd(&pub.hist_coarse[bn >> 5], 1);
                }
            }
            cluster.sync();  // every split's histogram is complete
            if (warp == 0) {
                // coarse bins (32 fine bins each), two per lane, descending, summed over the splits
                int ca = 0, cb = 0;
#pragma unroll
                for (int r = 0; r < kMaxSplits; ++r) {
                    if (r < S) {
                        const SelPub* rp = cluster.map_shared_rank(&pub, r);
                        ca += rp->hist_coarse[63 - 2 * lane];
                        cb += rp->hist_coarse[62 - 2 * lane];
                    }
                }
                int incl = ca + cb;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int y = __shfl_up_sync(full, incl, o);
                    if (lane >= o) incl += y;
                }
                const int need_here = beta - above;
                const unsigned hit = __ballot_sync(full, incl >= need_here);
                const int f = __ffs(hit) - 1;
                const int ex_f = __shfl_sync(full, incl - ca - cb, f), ca_f = __shfl_sync(full, ca, f);
                const bool upper = ex_f + ca_f >= need_here;
                const int cbin = upper ? 63 - 2 * f : 62 - 2 * f;
                const int above_c = upper ? ex_f : ex_f + ca_f;
                // the 32 fine bins of that coarse bin, descending by lane
                const int fb = cbin * 32 + 31 - lane;
                int hcnt = 0;
#pragma unroll
                for (int r = 0; r < kMaxSplits; ++r)
                    if (r < S) hcnt += cluster.map_shared_rank(&pub, r)->hist[fb];
                int fin = hcnt;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int y = __shfl_up_sync(full, fin, o);
                    if (lane >= o) fin += y;
                }
                const unsigned fhit = __ballot_sync(full, above_c + fin >= need_here);
                const int ff = __ffs(fhit) - 1;
                const int fin_f = __shfl_sync(full, fin, ff), h_f = __shfl_sync(full, hcnt, ff);
                if (lane == 0) {
                    sl.g[3] = cbin * 32 + 31 - ff;
                    sl.g[4] = above + above_c + fin_f - h_f;
                    sl.g[5] = h_f;
                }
            }
            __syncthreads();
            const int bstar = sl.g[3], above_new = sl.g[4], bcnt = sl.g[5];
            if (bcnt <= kSelCand) {
                mode = 1;
                above = above_new;
                need = beta - above;
                // keys above the range or in a higher bin are taken; the boundary bin's keys are candidates
                int nc = 0;
                for (int i = i0; i < i1; ++i) {
                    const uint32_t v = s_keys[i];
                    nc += v != 0u && v >= lo && v <= hi && bin_of(v) == bstar;
                }
                int tot;
                int pc = block_exclusive_scan(nc, sl.warp, tot);
                for (int i = i0; i < i1; ++i) {
                    const uint32_t v = s_keys[i];
                    if (v == 0u) continue;
                    if (v > hi || (v >= lo && bin_of(v) > bstar)) mark(i);
                    else if (v >= lo && bin_of(v) == bstar) {
                        pub.cand_key[pc] = v;
                        pub.cand_g[pc] = g0 + i;
                        ++pc;
                    }
                }
                if (tid == 0) pub.n_cand = tot;
                break;
            }
            // crowded boundary bin: continue inside its exact key range
            uint32_t bmx = 0u, bmn = 0xFFFFFFFFu;
            for (int i = tid; i < n; i += kThreads) {
                const uint32_t v = s_keys[i];
                if (v != 0u && v >= lo && v <= hi && bin_of(v) == bstar) { bmx = max(bmx, v); bmn = min(bmn, v); }
            }
            bmx = __reduce_max_sync(full, bmx);
            bmn = __reduce_min_sync(full, bmn);
            if (lane == 0) { sl.red[1][warp] = bmx; sl.red[2][warp] = bmn; }
            __syncthreads();
            if (tid == 0) {
                uint32_t hx = 0u, lx = 0xFFFFFFFFu;
#pragma unroll
                for (int w = 0; w < kThreads / 32; ++w) { hx = max(hx, sl.red[1][w]); lx = min(lx, sl.red[2][w]); }
                pub.bmax = hx; pub.bmin = lx;
            }
            cluster.sync();  // also: every split is done reading this level's histograms
            if (warp == 0) {
                uint32_t hx = 0u, lx = 0xFFFFFFFFu;
                if (lane < S) {
                    const SelPub* rp = cluster.map_shared_rank(&pub, lane);
                    hx = rp->bmax; lx = rp->bmin;
                }
                hx = __reduce_max_sync(full, hx);
                lx = __reduce_min_sync(full, lx);
                if (lane == 0) { sl.g[6] = (int)hx; sl.g[7] = (int)lx; }
            }
            __syncthreads();
            hi = (uint32_t)sl.g[6];
            lo = (uint32_t)sl.g[7];
            above = above_new;
        }
    }

    if (mode == 1) {
        cluster.sync();  // every split's candidates are published
        if (warp == 0) {
            // the candidates of all splits, one per lane, in split (= group) order
            const int ncr = lane < S ? cluster.map_shared_rank(&pub, lane)->n_cand : 0;
            int cpre = ncr;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(full, cpre, o);
                if (lane >= o) cpre += y;
            }
            const int ctot = __shfl_sync(full, cpre, 31);
            int r = 0;
            for (int j = 0; j < S; ++j) r += __shfl_sync(full, cpre, j) <= lane;
            const int start = __shfl_sync(full, cpre - ncr, min(r, 31));
            uint32_t ck = 0u;
            int cg = -1;
            if (lane < ctot) {
                const SelPub* rp = cluster.map_shared_rank(&pub, r);
                ck = rp->cand_key[lane - start];
                cg = rp->cand_g[lane - start];
            }
            int rank = 0;
            for (int j = 0; j < ctot; ++j) {
                const uint32_t kj = __shfl_sync(full, ck, j);
                const int gj = __shfl_sync(full, cg, j);
                rank += (kj > ck) || (kj == ck && gj < cg);
            }
            if (lane < ctot && rank < need && r == s) mark(cg - g0);
        }
    } else if (mode == 2) {
        // keys above kstar are taken, then the first `need` keys equal to kstar in group order
        int neq = 0;
        for (int i = i0; i < i1; ++i) neq += s_keys[i] == kstar;
        int tot;
        int eq_before = block_exclusive_scan(neq, sl.warp, tot);
        if (tid == 0) pub.n_eq = tot;
        cluster.sync();  // every split's count of equal keys is published
        if (warp == 0) {
            int t = lane < s ? cluster.map_shared_rank(&pub, lane)->n_eq : 0;
            t = __reduce_add_sync(full, t);
            if (lane == 0) sl.g[0] = t;
        }
        __syncthreads();
        const int take = min(max(need - sl.g[0], 0), tot);
        for (int i = i0; i < i1; ++i) {
            const uint32_t v = s_keys[i];
            if (v > kstar) mark(i);
            else if (v == kstar) {
                if (eq_before < take) mark(i);
                ++eq_before;
            }
        }
    } else {
        for (int i = tid; i < n; i += kThreads)
            if (s_keys[i] != 0u) mark(i);
    }
    __syncthreads();

    // this split's selected groups, ascending, then the concatenation over the splits
    {
        int c = 0;
        for (int i = i0; i < i1; ++i) c += (s_mark[i >> 5] >> (i & 31)) & 1u;
        int tot;
        int p = block_exclusive_scan(c, sl.warp, tot);
        for (int i = i0; i < i1; ++i) {
            if ((s_mark[i >> 5] >> (i & 31)) & 1u) {
                if (p < HSQ_MAX_BETA) pub.mine[p] = g0 + i;
                ++p;
            }
        }
        if (tid == 0) pub.n_mine = min(tot, beta);
    }
    cluster.sync();  // every split's list is published
    if (warp == 0) {
        const int nm = lane < S ? cluster.map_shared_rank(&pub, lane)->n_mine : 0;
        int incl = nm;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(full, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane < S) sl.off[lane + 1] = incl;
        if (lane == 0) sl.off[0] = 0;
    }
    __syncthreads();
    const int total = min(sl.off[S], beta);
    for (int i = tid; i < beta; i += kThreads) {
        int g = -1;
        if (i < total) {
            int r = 0;
            while (sl.off[r + 1] <= i) ++r;
            g = cluster.map_shared_rank(&pub, r)->mine[i - sl.off[r]];
        }
        s_sel[i] = g;
    }
    __syncthreads();
}

template <int R, int N, bool kRoute>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(CacheView c, DecodeArgs a, Tables tb) {
    namespace cgx = cooperative_groups;
    extern __shared__ __align__(16) uint8_t s_dyn[];
    __shared__ __align__(16) float s_cb[hsq::kCodebookFloats];
    __shared__ __align__(16) float s_qt[R][kDim];
    __shared__ __align__(16) float s_qr[R][kDim];
    __shared__ __align__(16) float s_ppart[R][hsq::kPartStride];  // this split's partial, read by the others
    __shared__ SelPub s_pub;
    __shared__ SelLocal s_sl;

    constexpr int RB = N * 136;
    constexpr int kBatchRecs = kFetchBatchBytes / RB;
    constexpr int kRecChunks = RB / 16;

    cgx::cluster_group cluster = cgx::this_cluster();
    const int S = (int)cluster.num_blocks();
    const int s = (int)cluster.block_rank();
    const int bh = blockIdx.y, b = bh / c.Hkv, h = bh % c.Hkv;
    const int tid = threadIdx.x, hw = tid >> 4, l = hlane(), lane = tid & 31, warp = tid >> 5;
    const unsigned m = half_mask();
    const unsigned full = 0xffffffffu;
    const int fl = a.flags;
    const DecodeLayout L = decode_layout<R, N>(c.G, c.T, S, c.max_l1, c.beta, kRoute, fl);

    const int g0 = (int)((long long)c.G * s / S), g1 = (int)((long long)c.G * (s + 1) / S);
    const int n2 = g1 - g0;
    const int cnt1 = min(__ldg(c.l1_count + b), c.max_l1);
    const int e0 = (int)((long long)cnt1 * s / S), e1 = (int)((long long)cnt1 * (s + 1) / S);
    const int n1 = e1 - e0;
    const int f0 = (int)((long long)c.beta * s / S), f1 = (int)((long long)c.beta * (s + 1) / S);
    const int nfetch = f1 - f0;

    // inputs: staged copies in shared memory, or read in place
    const uint8_t* g_l2k = c.l2_kc + ((size_t)bh * c.G + g0) * 48;
    const uint8_t* g_l2v = c.l2_vc + ((size_t)bh * c.G + g0) * 48;
    const float* g_l2kn = c.l2_kn + (size_t)bh * c.G + g0;
    const float* g_l2vn = c.l2_vn + (size_t)bh * c.G + g0;
    const uint8_t* g_cnt = c.l2_cnt + (size_t)b * c.G + g0;
    const uint8_t* g_l1k = c.l1_kc + ((size_t)bh * c.max_l1 + e0) * 64;
    const uint8_t* g_l1v = c.l1_vc + ((size_t)bh * c.max_l1 + e0) * 64;
    const float* g_l1kn = c.l1_kn + (size_t)bh * c.max_l1 + e0;
    const float* g_l1vn = c.l1_vn + (size_t)bh * c.max_l1 + e0;
    const uint32_t* g_bitmap = c.l1_bitmap + (size_t)b * c.W;
    const bool st2 = fl & kStageL2, st1 = fl & kStageL1, stb = fl & kStageBitmap, keep = fl & kKeepLogits;
    const uint8_t* p_l2k = st2 ? s_dyn + L.l2k : g_l2k;
    const uint8_t* p_l2v = st2 ? s_dyn + L.l2v : g_l2v;
    const float* p_l2kn = st2 ? reinterpret_cast<const float*>(s_dyn + L.l2kn) : g_l2kn;
    const float* p_l2vn = st2 ? reinterpret_cast<const float*>(s_dyn + L.l2vn) : g_l2vn;
    const uint8_t* p_cnt = st2 ? s_dyn + L.cnt : g_cnt;
    const uint8_t* p_l1k = st1 ? s_dyn + L.l1k : g_l1k;
    const uint8_t* p_l1v = st1 ? s_dyn + L.l1v : g_l1v;
    const float* p_l1kn = st1 ? reinterpret_cast<const float*>(s_dyn + L.l1kn) : g_l1kn;
    const float* p_l1vn = st1 ? reinterpret_cast<const float*>(s_dyn + L.l1vn) : g_l1vn;
    const uint32_t* p_bitmap = stb ? reinterpret_cast<const uint32_t*>(s_dyn + L.bitmap) : g_bitmap;
    float* s_logit = reinterpret_cast<float*>(s_dyn + L.logit);
    uint32_t* s_keys = reinterpret_cast<uint32_t*>(s_dyn + L.keys);
    int* s_sel = reinterpret_cast<int*>(s_dyn + L.sel);
    uint32_t* s_mask = reinterpret_cast<uint32_t*>(s_dyn + L.mask);
    float* s_lev = reinterpret_cast<float*>(s_dyn + L.lev);
    float* s_b0 = reinterpret_cast<float*>(s_dyn + L.b0);
    float* s_off = reinterpret_cast<float*>(s_dyn + L.off);
    float* s_base = reinterpret_cast<float*>(s_dyn + L.base);
    uint32_t* s_rbits = reinterpret_cast<uint32_t*>(s_dyn + L.rbits);
    uint8_t* s_rec = s_dyn + L.rec;

    // 1. stage the device-resident inputs of this split
    if (st2) {
        stage16(s_dyn + L.l2k, g_l2k, n2 * 48);
        stage16(s_dyn + L.l2v, g_l2v, n2 * 48);
        stage4(reinterpret_cast<float*>(s_dyn + L.l2kn), g_l2kn, n2);
        stage4(reinterpret_cast<float*>(s_dyn + L.l2vn), g_l2vn, n2);
        for (int i = tid; i < n2; i += kThreads) s_dyn[L.cnt + i] = __ldg(g_cnt + i);
    }
    if (st1) {
        stage16(s_dyn + L.l1k, g_l1k, n1 * 64);
        stage16(s_dyn + L.l1v, g_l1v, n1 * 64);
        stage4(reinterpret_cast<float*>(s_dyn + L.l1kn), g_l1kn, n1);
        stage4(reinterpret_cast<float*>(s_dyn + L.l1vn), g_l1vn, n1);
    }
    if (stb) stage4(reinterpret_cast<float*>(s_dyn + L.bitmap), reinterpret_cast<const float*>(g_bitmap), c.W);
    if (tid < hsq::kCodebookFloats / 4) cp_async16(s_cb + 4 * tid, tb.cb + 4 * tid);
    // RoPE rows: level k row j = hi[j * 16^k] (angle 256 j 16^k omega), b0 row j = lo[N j], off row n = lo[n]
    const int n_hi = (tb.max_pos + 255) / 256;
    for (int i = tid; i < L.nlev * 16 * 32; i += kThreads) {
        const int rowi = i >> 5, k = rowi >> 4, j = rowi & 15;
        const int src = j << (4 * k);
        if (src < n_hi) cp_async16(s_lev + 4 * i, tb.rope_hi + (size_t)src * kDim + 4 * (i & 31));
    }
    for (int i = tid; i < L.nb0 * 32; i += kThreads)
        cp_async16(s_b0 + 4 * i, tb.rope_lo + (size_t)(N * (i >> 5)) * kDim + 4 * (i & 31));
    stage16(s_off, tb.rope_lo, N * kDim * 4);
    for (int i = tid; i < (L.span + 31) / 32; i += kThreads) s_mask[i] = 0u;
    float sg[8];
    load_signs_global(sg, c.signs);

    // 2. query heads of this KV head: RoPE'd (original frame) and rotated
    const int pos = checked_pos(__ldg(a.pos + b), tb, a.err);
    if (hw < R) {
        const int j = h * R + hw;
        float x[8];
        load_f32x8(a.q + ((size_t)b * c.Hq + j) * kDim, x);
        rope(x, pos, tb);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            s_qr[hw][4 * l + k] = x[k];
            s_qr[hw][64 + 4 * l + k] = x[4 + k];
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] *= sg[i];
        fwht(x, m);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            s_qt[hw][4 * l + k] = x[k] * kRsqrtD;
            s_qt[hw][64 + 4 * l + k] = x[4 + k] * kRsqrtD;
        }
    }
    cp_async_wait_all();
    __syncthreads();

    const float* c4 = s_cb;
    const float* c3 = s_cb + 32;
    float qt[R][8];
#pragma unroll
    for (int j = 0; j < R; ++j) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            qt[j][k] = s_qt[j][4 * l + k];
            qt[j][4 + k] = s_qt[j][64 + 4 * l + k];
        }
    }
    // log2-domain logits of L2 groups i and ib against every query head
    auto l2_logits = [&](int i, int ib, float xa[R], float xb[R]) {
        float va[8], vb[8];
        unpack3_smem(p_l2k + i * 48, c3, 1.0f, va);
        unpack3_smem(p_l2k + ib * 48, c3, 1.0f, vb);
        const float kna = p_l2kn[i], knb = p_l2kn[ib];
#pragma unroll
        for (int j = 0; j < R; ++j) {
            float da = 0.f, db = 0.f;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                da = fmaf(qt[j][k], va[k], da);
                db = fmaf(qt[j][k], vb[k], db);
            }
            xa[j] = kna * half_sum(da, m) * kLogitScaleLog2;
            xb[j] = knb * half_sum(db, m) * kLogitScaleLog2;
        }
    };
    if (kRoute || keep) {
        float gq[8];
        if (kRoute) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                float s0 = 0.f, s1 = 0.f;
#pragma unroll
                for (int jj = 0; jj < R; ++jj) {
                    s0 += s_qt[jj][4 * l + k];
                    s1 += s_qt[jj][64 + 4 * l + k];
                }
                gq[k] = s0;
                gq[4 + k] = s1;
            }
        }
        // two groups per half-warp per iteration (independent instruction streams)
        for (int i = hw; i < n2; i += 2 * kHalves) {
            const int ib = i + kHalves;
            const bool hb = ib < n2;
            const int ibs = hb ? ib : i;
            if (kRoute) {
                float va[8], vb[8];
                unpack3_smem(p_l2k + i * 48, c3, 1.0f, va);
                unpack3_smem(p_l2k + ibs * 48, c3, 1.0f, vb);
                float da = 0.f, db = 0.f;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    da = fmaf(gq[k], va[k], da);
                    db = fmaf(gq[k], vb[k], db);
                }
                da = half_sum(da, m);
                db = half_sum(db, m);
                if (l == 0) {
                    s_keys[i] = p_cnt[i] > 0 ? ordered_key(p_l2kn[i] * da) : 0u;
                    if (hb) s_keys[ib] = p_cnt[ib] > 0 ? ordered_key(p_l2kn[ib] * db) : 0u;
                }
            }
            if (keep) {
                float xa[R], xb[R];
                l2_logits(i, ibs, xa, xb);
                if (l == 0) {
#pragma unroll
                    for (int j = 0; j < R; ++j) {
                        s_logit[i * R + j] = xa[j];
                        if (hb) s_logit[ib * R + j] = xb[j];
                    }
                }
            }
        }
    }

    // 3. the selection of this (b, h)
    if (kRoute) {
        __syncthreads();  // this split's keys are written
        cluster_select(s_keys, n2, g0, c.beta, s_sel, s_mask, s_pub, s_sl);
        if (s == 0)
            for (int i = tid; i < c.beta; i += kThreads) a.sel[(size_t)bh * c.beta + i] = s_sel[i];
    } else {
        for (int i = tid; i < c.beta; i += kThreads) s_sel[i] = valid_sel(a.sel + (size_t)bh * c.beta, i, c.G, a.err);
        __syncthreads();
        for (int i = tid; i < c.beta; i += kThreads) {
            const int g = s_sel[i];
            if (g >= g0 && g < g1) atomicOr(&s_mask[(g - g0) >> 5], 1u << ((g - g0) & 31));
        }
    }

    // 4. gather this split's records; meanwhile L1 tokens and unselected summaries
    uint4 pre[kMaxFetchChunksPerThread];
    auto issue = [&](int r0, int nrec) {
#pragma unroll
        for (int k = 0; k < kMaxFetchChunksPerThread; ++k) {
            const int ch = tid + k * kThreads;
            pre[k] = make_uint4(0, 0, 0, 0);
            if (ch < nrec * kRecChunks) {
                const int rec = ch / kRecChunks, off = ch - rec * kRecChunks;
                const int i = r0 + rec;
                const int g = s_sel[i];
                if (g >= 0) {
                    const uint8_t* base = a.from_staging ? c.staging + ((size_t)bh * c.beta + i) * RB
                                                         : c.l3 + ((size_t)bh * c.G + g) * RB;
                    pre[k] = __ldcg(reinterpret_cast<const uint4*>(base) + off);
                }
            }
        }
    };
    // per record: cos/sin of its base angle g N omega (staged rows only) and its L1 bits
    auto meta = [&](int r0, int nrec) {
        if (hw < nrec) {
            const int g = s_sel[r0 + hw];
            if (g >= 0) {
                const int p0 = g * N;
                const float* br = s_b0 + ((p0 & 255) / N) * kDim;
                float4 cs = *reinterpret_cast<const float4*>(br + 4 * l);
                float4 sn = *reinterpret_cast<const float4*>(br + 64 + 4 * l);
                int rest = p0 >> 8;
                for (int k = 0; rest > 0; ++k, rest >>= 4) {
                    const int j = rest & 15;
                    if (j) {
                        const float* lr = s_lev + (k * 16 + j) * kDim;
                        angle_add4(cs, sn, *reinterpret_cast<const float4*>(lr + 4 * l),
                                   *reinterpret_cast<const float4*>(lr + 64 + 4 * l));
                    }
                }
                *reinterpret_cast<float4*>(s_base + hw * kDim + 4 * l) = cs;
                *reinterpret_cast<float4*>(s_base + hw * kDim + 64 + 4 * l) = sn;
                if (l == 0)
                    s_rbits[hw] = (p_bitmap[p0 >> 5] >> (p0 & 31)) & ((N == 32) ? 0xFFFFFFFFu : ((1u << N) - 1u));
            }
        }
    };
    const int nb0 = min(nfetch, kBatchRecs);
    if (nb0 > 0) {
        issue(f0, nb0);
        meta(f0, nb0);
    }
    __syncthreads();  // s_mask complete (kRoute: marked by the selection)

    Softmax<R> sm;
    sm.init();
    {
        auto entry = [&](int e, float x[R], float vv[8]) {
            const uint16_t* kr = reinterpret_cast<const uint16_t*>(p_l1k + e * 64);
            const uint16_t* vr = reinterpret_cast<const uint16_t*>(p_l1v + e * 64);
            float kv[8];
            unpack4(kr[l], kr[16 + l], c4, p_l1kn[e], kv);
            unpack4(vr[l], vr[16 + l], c4, p_l1vn[e], vv);
#pragma unroll
            for (int j = 0; j < R; ++j) {
                float d = 0.f;
#pragma unroll
                for (int k = 0; k < 8; ++k) d = fmaf(qt[j][k], kv[k], d);
                x[j] = half_sum(d, m) * kLogitScaleLog2;
            }
        };
        for (int e = hw; e < n1; e += 2 * kHalves) {
            const int eb = e + kHalves;
            const bool hb = eb < n1;
            float xa[R], xb[R], va[8], vb[8];
            entry(e, xa, va);
            entry(hb ? eb : e, xb, vb);
            sm.add2(xa, va, true, xb, vb, hb);
        }
    }
    for (int i = hw; i < n2; i += 2 * kHalves) {
        const int ib = i + kHalves;
        const int ibs = ib < n2 ? ib : i;
        const bool oka = p_cnt[i] > 0 && !((s_mask[i >> 5] >> (i & 31)) & 1u);
        const bool okb = ib < n2 && p_cnt[ibs] > 0 && !((s_mask[ibs >> 5] >> (ibs & 31)) & 1u);
        if (!oka && !okb) continue;
        float va[8], vb[8], xa[R], xb[R];
        unpack3_smem(p_l2v + i * 48, c3, p_l2vn[i], va);
        unpack3_smem(p_l2v + ibs * 48, c3, p_l2vn[ibs], vb);
        if (keep) {
#pragma unroll
            for (int j = 0; j < R; ++j) {
                xa[j] = s_logit[i * R + j];
                xb[j] = s_logit[ibs * R + j];
            }
        } else {
            l2_logits(i, ibs, xa, xb);
        }
        sm.add2(xa, va, oka, xb, vb, okb);
    }

    // 5. recovered tokens of the selected groups
    if (nfetch > 0) {
        float qr[R][8];
#pragma unroll
        for (int j = 0; j < R; ++j) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                qr[j][k] = s_qr[j][4 * l + k];
                qr[j][4 + k] = s_qr[j][64 + 4 * l + k];
            }
        }
        for (int r0 = f0; r0 < f1; r0 += kBatchRecs) {
            const int nb = min(kBatchRecs, f1 - r0);
            __syncthreads();  // previous batch consumed, this batch's meta written
#pragma unroll
            for (int k = 0; k < kMaxFetchChunksPerThread; ++k) {
                const int ch = tid + k * kThreads;
                if (ch < nb * kRecChunks) reinterpret_cast<uint4*>(s_rec)[ch] = pre[k];
            }
            __syncthreads();
            const bool more = r0 + kBatchRecs < f1;
            if (more) issue(r0 + kBatchRecs, min(kBatchRecs, f1 - r0 - kBatchRecs));
            // one recovered token: validity, logits against the RoPE'd queries, rotated-frame value
            auto token = [&](int u, float x[R], float vv[8]) -> bool {
                const int rec = u / N, n = u - rec * N;
                const int g = s_sel[r0 + rec];
                const int t = g * N + n;
                const bool ok = g >= 0 && t < c.T && !((s_rbits[rec] >> n) & 1u);
                const uint8_t* rp = s_rec + rec * RB;
                const float* norms = reinterpret_cast<const float*>(rp + N * 128);
                const uint16_t* kr = reinterpret_cast<const uint16_t*>(rp + n * 64);
                const uint16_t* vr = reinterpret_cast<const uint16_t*>(rp + N * 64 + n * 64);
                float kv[8];
                unpack4(kr[l], kr[16 + l], c4, 1.0f, kv);
                fwht(kv, m);
                const float kn = norms[n] * kRsqrtD;
#pragma unroll
                for (int i = 0; i < 8; ++i) kv[i] *= sg[i] * kn;
                {   // RoPE at t = g N + n: base angle (per record) plus offset n omega
                    float4 cs = *reinterpret_cast<const float4*>(s_base + rec * kDim + 4 * l);
                    float4 sn = *reinterpret_cast<const float4*>(s_base + rec * kDim + 64 + 4 * l);
                    angle_add4(cs, sn, *reinterpret_cast<const float4*>(s_off + n * kDim + 4 * l),
                               *reinterpret_cast<const float4*>(s_off + n * kDim + 64 + 4 * l));
                    const float cv[4] = {cs.x, cs.y, cs.z, cs.w}, sv[4] = {sn.x, sn.y, sn.z, sn.w};
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float lo = kv[k], hi = kv[4 + k];
                        kv[k] = fmaf(lo, cv[k], -hi * sv[k]);
                        kv[4 + k] = fmaf(hi, cv[k], lo * sv[k]);
                    }
                }
                unpack4(vr[l], vr[16 + l], c4, norms[N + n], vv);
#pragma unroll
                for (int j = 0; j < R; ++j) {
                    float d = 0.f;
#pragma unroll
                    for (int i = 0; i < 8; ++i) d = fmaf(qr[j][i], kv[i], d);
                    x[j] = half_sum(d, m) * kLogitScaleLog2;
                }
                return ok;
            };
            for (int u = hw; u < nb * N; u += 2 * kHalves) {
                const int ub = u + kHalves;
                const bool hb = ub < nb * N;
                float xa[R], xb[R], va[8], vb[8];
                const bool oka = token(u, xa, va);
                const bool okb = token(hb ? ub : u, xb, vb) && hb;
                sm.add2(xa, va, oka, xb, vb, okb);
            }
            if (more) {
                __syncthreads();
                meta(r0 + kBatchRecs, min(kBatchRecs, f1 - r0 - kBatchRecs));
            }
        }
    }

    // 6. merge the two halves of each warp, then the warps, into this split's published partial
    __syncwarp();
#pragma unroll
    for (int j = 0; j < R; ++j) {
        const float mo = __shfl_xor_sync(full, sm.m[j], 16);
        const float lo = __shfl_xor_sync(full, sm.l[j], 16);
        const float M = fmaxf(sm.m[j], mo);
        const float ws = merge_weight(sm.m[j], M), wo = merge_weight(mo, M);
        sm.l[j] = sm.l[j] * ws + lo * wo;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float ao = __shfl_xor_sync(full, sm.acc[j][i], 16);
            sm.acc[j][i] = sm.acc[j][i] * ws + ao * wo;
        }
        sm.m[j] = M;
    }
    __syncthreads();  // the record staging area becomes the warp-partial area
    float* s_part = reinterpret_cast<float*>(s_rec);  // [8 warps][R][132]
    if ((tid & 16) == 0) {
#pragma unroll
        for (int j = 0; j < R; ++j) {
            float* p = s_part + ((size_t)warp * R + j) * hsq::kPartStride;
            *reinterpret_cast<float4*>(p + 4 * l) = make_float4(sm.acc[j][0], sm.acc[j][1], sm.acc[j][2], sm.acc[j][3]);
            *reinterpret_cast<float4*>(p + 64 + 4 * l) = make_float4(sm.acc[j][4], sm.acc[j][5], sm.acc[j][6], sm.acc[j][7]);
            if (l == 0) { p[128] = sm.m[j]; p[129] = sm.l[j]; }
        }
    }
    __syncthreads();
    if (tid < R * 32) {
        const int j = tid >> 5, q4 = tid & 31;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) M = fmaxf(M, s_part[((size_t)w * R + j) * hsq::kPartStride + 128]);
        float Lsum = 0.f;
        float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) {
            const float* p = s_part + ((size_t)w * R + j) * hsq::kPartStride;
            const float wt = merge_weight(p[128], M);
            const float4 v = *reinterpret_cast<const float4*>(p + 4 * q4);
            Lsum += p[129] * wt;
            A.x += v.x * wt; A.y += v.y * wt; A.z += v.z * wt; A.w += v.w * wt;
        }
        *reinterpret_cast<float4*>(&s_ppart[j][4 * q4]) = A;
        if (q4 == 0) { s_ppart[j][128] = M; s_ppart[j][129] = Lsum; }
    }
    cluster.sync();  // every split's partial is published

    // query head j is merged by split j mod S (warp w: head s + w S), then rotated back by one half-warp
    float* s_o = s_qr[0];  // [R][128]; the RoPE'd queries are no longer needed
    const int nmine = (R - s + S - 1) / S;
    if (warp < nmine) {
        const int j = s + warp * S;
        float mr = -INFINITY, lr = 0.f;
        if (lane < S) {
            const float* pp = cluster.map_shared_rank(&s_ppart[j][0], lane);
            mr = pp[128];
            lr = pp[129];
        }
        const float M = warp_max(mr);
        const float wr = merge_weight(mr, M);
        const float Lsum = warp_sum(lr * wr);
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int r = 0; r < kMaxSplits; ++r) {
            const float wt = __shfl_sync(full, wr, r);
            if (r < S) {
                const float4 x = *reinterpret_cast<const float4*>(cluster.map_shared_rank(&s_ppart[j][0], r) + 4 * lane);
                o.x += x.x * wt; o.y += x.y * wt; o.z += x.z * wt; o.w += x.w * wt;
            }
        }
        const float inv = Lsum > 0.f ? 1.0f / Lsum : 0.f;
        *reinterpret_cast<float4*>(s_o + j * kDim + 4 * lane) = make_float4(o.x * inv, o.y * inv, o.z * inv, o.w * inv);
    }
    __syncthreads();
    if (hw < 2 * nmine && (hw & 1) == 0) {
        const int j = s + (hw >> 1) * S;
        float o[8];
        load_f32x8_smem(s_o + j * kDim, o);
        fwht(o, m);  // back to the original frame: Pi^T o = diag(s) H o / sqrt(d)
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i] *= sg[i] * kRsqrtD;
        store_f32x8(a.out + ((size_t)b * c.Hq + h * R + j) * kDim, o);
    }
    cluster.sync();  // this split's shared memory stays alive until every reader is done
}

}  // namespace

// ===========================================================================
// Host side: context and entry points.
// ===========================================================================

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
    // decode launch plan per cache shape: cluster size S (0 = cannot launch) and staging flags
    struct Plan { int B, T, route, S, flags; };
    std::vector<Plan> plans;
    std::string last_error;
};

namespace {

hsq_status fail(hsq_ctx* ctx, hsq_status st, const std::string& msg) {
    if (ctx) ctx->last_error = msg;
    hsq::set_process_error(msg);
    return st;
}

hsq_status cuda_fail(hsq_ctx* ctx, cudaError_t e, const char* where) {
    return fail(ctx, HSQ_ERR_CUDA, std::string(where) + ": " + cudaGetErrorString(e));
}

#define HSQ_CUDA(ctx, call)                                   \
    do {                                                      \
        cudaError_t e_ = (call);                              \
        if (e_ != cudaSuccess) return cuda_fail(ctx, e_, #call); \
    } while (0)

bool r_supported(int r) { return r == 1 || r == 2 || r == 4 || r == 5 || r == 8; }

CacheView make_view(const hsq_ctx* ctx, const hsq_cache* c) {
    CacheView v{};
    v.B = c->B; v.T = c->T; v.N = ctx->cfg.group_n; v.G = hsq::groups_of(c->T, v.N);
    v.Hkv = ctx->cfg.n_kv_heads; v.Hq = ctx->cfg.n_q_heads; v.beta = ctx->cfg.beta;
    v.max_l1 = ctx->cfg.max_l1; v.W = hsq::bitmap_words(c->T);
    v.l1_kc = c->l1_kc; v.l1_vc = c->l1_vc; v.l1_kn = c->l1_kn; v.l1_vn = c->l1_vn;
    v.l1_pos = c->l1_pos; v.l1_count = c->l1_count;
    v.l2_kc = c->l2_kc; v.l2_vc = c->l2_vc; v.l2_kn = c->l2_kn; v.l2_vn = c->l2_vn; v.l2_cnt = c->l2_cnt;
    v.l3 = c->l3; v.l1_bitmap = c->l1_bitmap; v.signs = c->signs; v.staging = c->staging;
    return v;
}

Tables make_tables(const hsq_ctx* ctx) {
    Tables t{};
    t.cb = ctx->d_cb; t.rope_hi = ctx->d_rope_hi; t.rope_lo = ctx->d_rope_lo; t.max_pos = ctx->cfg.max_pos;
    return t;
}

// The dynamic shared-memory ceiling is a property of the kernel (per device),
// shared by every context of the process: only ever raise it.
std::mutex g_smem_mu;
std::vector<std::pair<std::pair<const void*, int>, size_t>> g_smem_limits;

cudaError_t raise_smem_limit(const void* fn, int device, size_t bytes) {
    std::lock_guard<std::mutex> lk(g_smem_mu);
    for (auto& e : g_smem_limits) {
        if (e.first.first == fn && e.first.second == device) {
            if (e.second >= bytes) return cudaSuccess;
            cudaError_t err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
            if (err == cudaSuccess) e.second = bytes;
            return err;
        }
    }
    cudaError_t err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (err == cudaSuccess) g_smem_limits.push_back({{fn, device}, bytes});
    return err;
}

template <int V>
using IC = std::integral_constant<int, V>;

// Calls f(IC<R>{}, IC<N>{}) for the context's head ratio and group size.
template <class F>
hsq_status dispatch_rn(int r, int n, F&& f) {
    const bool n8 = n == 8;
    switch (r) {
        case 1: return n8 ? f(IC<1>{}, IC<8>{}) : f(IC<1>{}, IC<16>{});
        case 2: return n8 ? f(IC<2>{}, IC<8>{}) : f(IC<2>{}, IC<16>{});
        case 4: return n8 ? f(IC<4>{}, IC<8>{}) : f(IC<4>{}, IC<16>{});
        case 5: return n8 ? f(IC<5>{}, IC<8>{}) : f(IC<5>{}, IC<16>{});
        case 8: return n8 ? f(IC<8>{}, IC<8>{}) : f(IC<8>{}, IC<16>{});
    }
    return HSQ_ERR_UNSUPPORTED;
}

// Kernels allowed to run in 16-CTA clusters (the portable limit is 8).
std::vector<std::pair<const void*, int>> g_big_clusters;

cudaError_t allow_big_clusters(const void* fn, int device) {
    std::lock_guard<std::mutex> lk(g_smem_mu);
    for (auto& e : g_big_clusters)
        if (e.first == fn && e.second == device) return cudaSuccess;
    cudaError_t err = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (err == cudaSuccess) g_big_clusters.push_back({fn, device});
    return err;
}

cudaLaunchConfig_t decode_config(int S, int bh, size_t smem, cudaStream_t st, cudaLaunchAttribute* at) {
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(S, bh, 1);
    lc.blockDim = dim3(kThreads, 1, 1);
    lc.dynamicSmemBytes = smem;
    lc.stream = st;
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = S;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    lc.attrs = at;
    lc.numAttrs = 1;
    return lc;
}

// Cluster size of the decode kernel for B sequences of T tokens: the largest
// S <= 16 whose B * Hkv clusters are all resident at once (one wave); when no
// S gives one wave, S = 1 (least per-head overhead across waves).  A fixed
// n_splits is an upper bound.  Inputs that do not fit in shared memory are
// left in global memory, dropping first the kept L2 logits, then the L1
// slice, then the bitmap row, then the L2 slice.
template <int R, int N, bool kRoute>
hsq_ctx::Plan decode_plan(hsq_ctx* ctx, int B, int T) {
    for (const auto& e : ctx->plans)
        if (e.B == B && e.T == T && e.route == (int)kRoute) return e;
    const int G = hsq::groups_of(T, N);
    const int bh = B * ctx->cfg.n_kv_heads;
    const void* fn = (const void*)decode_kernel<R, N, kRoute>;
    hsq_ctx::Plan plan{B, T, (int)kRoute, 0, 0};
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, fn) == cudaSuccess && allow_big_clusters(fn, ctx->device) == cudaSuccess) {
        const size_t cap = (size_t)ctx->smem_optin > fa.sharedSizeBytes ? ctx->smem_optin - fa.sharedSizeBytes : 0;
        const int fixed = ctx->cfg.n_splits;
        const int s_hi = std::max(1, std::min(fixed > 0 ? fixed : kMaxSplits, std::max(G, 1)));
        static const int kFlagOrder[] = {kStageL2 | kKeepLogits | kStageL1 | kStageBitmap,
                                         kStageL2 | kStageL1 | kStageBitmap, kStageL2 | kStageBitmap, kStageL2, 0};
        for (int S = s_hi; S >= 1; --S) {
            int flags = -1;
            size_t smem = 0;
            for (int f : kFlagOrder) {
                smem = decode_layout<R, N>(G, T, S, ctx->cfg.max_l1, ctx->cfg.beta, kRoute, f).total;
                if (smem <= cap) { flags = f; break; }
            }
            if (flags < 0) continue;
            if (raise_smem_limit(fn, ctx->device, smem) != cudaSuccess) continue;
            cudaLaunchAttribute at[1];
            cudaLaunchConfig_t lc = decode_config(S, bh, smem, 0, at);
            int nc = 0;
            if (cudaOccupancyMaxActiveClusters(&nc, fn, &lc) != cudaSuccess || nc < 1) continue;
            plan.S = S;
            plan.flags = flags;
            if (fixed > 0 || nc >= bh) break;  // otherwise keep going down to S = 1
        }
    }
    cudaGetLastError();
    ctx->plans.push_back(plan);
    return plan;
}

template <int R, int N, bool kRoute>
hsq_status launch_decode(hsq_ctx* ctx, CacheView v, DecodeArgs a, const hsq_ctx::Plan& p, cudaStream_t st) {
    a.flags = p.flags;
    const DecodeLayout L = decode_layout<R, N>(v.G, v.T, p.S, v.max_l1, v.beta, kRoute, p.flags);
    const void* fn = (const void*)decode_kernel<R, N, kRoute>;
    cudaError_t e = raise_smem_limit(fn, ctx->device, L.total);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaFuncSetAttribute(decode)");
    cudaLaunchAttribute at[1];
    const cudaLaunchConfig_t lc = decode_config(p.S, v.B * v.Hkv, L.total, st, at);
    const Tables tb = make_tables(ctx);
    e = cudaLaunchKernelEx(&lc, decode_kernel<R, N, kRoute>, v, a, tb);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "decode launch");
    return HSQ_OK;
}

template <int R>
hsq_status launch_route(hsq_ctx* ctx, const CacheView& v, const RouteArgs& a, cudaStream_t st) {
    const unsigned smem = route_smem_bytes(v.G);
    cudaError_t e = raise_smem_limit((const void*)route_kernel<R>, ctx->device, smem);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaFuncSetAttribute(route)");
    dim3 grid((v.G + kRouteGroupsPerCta - 1) / kRouteGroupsPerCta, v.B * v.Hkv);
    route_kernel<R><<<grid, kThreads, smem, st>>>(v, a, make_tables(ctx));
    return HSQ_OK;
}

hsq_status dispatch_route(hsq_ctx* ctx, const CacheView& v, const RouteArgs& a, cudaStream_t st) {
    switch (ctx->r) {
        case 1: return launch_route<1>(ctx, v, a, st);
        case 2: return launch_route<2>(ctx, v, a, st);
        case 4: return launch_route<4>(ctx, v, a, st);
        case 5: return launch_route<5>(ctx, v, a, st);
        case 8: return launch_route<8>(ctx, v, a, st);
    }
    return HSQ_ERR_UNSUPPORTED;
}

hsq_status after_launch(hsq_ctx* ctx, const char* what) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(ctx, e, what);
    return HSQ_OK;
}

hsq_status check_common(hsq_ctx* ctx, const hsq_cache* cache) {
    if (!ctx) return fail(nullptr, HSQ_ERR_INVALID, "context is NULL");
    std::string why = hsq::check_cache_shape(&ctx->cfg, cache);
    if (!why.empty()) return fail(ctx, HSQ_ERR_INVALID, why);
    return HSQ_OK;
}

void free_ctx(hsq_ctx* c) {
    cudaFree(c->d_cb); cudaFree(c->d_rope_hi); cudaFree(c->d_rope_lo); cudaFree(c->d_scores);
    cudaFree(c->d_route_ctr); cudaFree(c->d_prefix); cudaFree(c->d_err);
    delete c;
}

}  // namespace

extern "C" {

hsq_status hsq_create(const hsq_config* cfg, hsq_ctx** out) {
    if (!out) return fail(nullptr, HSQ_ERR_INVALID, "out is NULL");
    *out = nullptr;
    std::string why = hsq::check_config(cfg);
    if (!why.empty()) return fail(nullptr, HSQ_ERR_INVALID, why);
    if (hsq::fault_mask() & HSQ_FAULT_ALLOC) return fail(nullptr, HSQ_ERR_NOMEM, "injected allocation failure");
    const int r = cfg->n_q_heads / cfg->n_kv_heads;
    if (!r_supported(r)) return fail(nullptr, HSQ_ERR_UNSUPPORTED, "r = Hq/Hkv must be 1, 2, 4, 5 or 8");

    hsq_ctx* c = new hsq_ctx();
    c->cfg = *cfg;
    c->r = r;
    auto bail = [&](cudaError_t e, const char* where) {
        hsq_status st = (e == cudaErrorMemoryAllocation) ? HSQ_ERR_NOMEM : HSQ_ERR_CUDA;
        std::string msg = std::string(where) + ": " + cudaGetErrorString(e);
        free_ctx(c);
        return fail(nullptr, st, msg);
    };
    cudaError_t e;
    if ((e = cudaGetDevice(&c->device)) != cudaSuccess) return bail(e, "cudaGetDevice");
    if ((e = cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->device)) != cudaSuccess)
        return bail(e, "cudaDeviceGetAttribute");
    if ((e = cudaDeviceGetAttribute(&c->smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, c->device)) !=
        cudaSuccess)
        return bail(e, "cudaDeviceGetAttribute");

    float cb[hsq::kCodebookFloats];
    hsq::device_codebook(cb);
    std::vector<float> hi, lo;
    hsq::rope_tables(cfg->rope_theta, cfg->max_pos, hi, lo);
    c->G_max = hsq::groups_of(cfg->max_ctx, cfg->group_n);
    c->W_max = hsq::bitmap_words(cfg->max_ctx);
    const size_t bh = (size_t)cfg->max_batch * cfg->n_kv_heads;

    if ((e = cudaMalloc(&c->d_cb, sizeof(cb))) != cudaSuccess) return bail(e, "cudaMalloc(codebook)");
    if ((e = cudaMalloc(&c->d_rope_hi, hi.size() * 4)) != cudaSuccess) return bail(e, "cudaMalloc(rope)");
    if ((e = cudaMalloc(&c->d_rope_lo, lo.size() * 4)) != cudaSuccess) return bail(e, "cudaMalloc(rope)");
    if ((e = cudaMalloc(&c->d_scores, bh * c->G_max * 4)) != cudaSuccess) return bail(e, "cudaMalloc(scores)");
    if ((e = cudaMalloc(&c->d_route_ctr, bh * 4)) != cudaSuccess) return bail(e, "cudaMalloc(counters)");
    if ((e = cudaMalloc(&c->d_prefix, (size_t)cfg->max_batch * c->W_max * 4)) != cudaSuccess)
        return bail(e, "cudaMalloc(prefix)");
    if ((e = cudaMalloc(&c->d_err, 4)) != cudaSuccess) return bail(e, "cudaMalloc(err)");
    if ((e = cudaMemcpy(c->d_cb, cb, sizeof(cb), cudaMemcpyHostToDevice)) != cudaSuccess) return bail(e, "upload");
    if ((e = cudaMemcpy(c->d_rope_hi, hi.data(), hi.size() * 4, cudaMemcpyHostToDevice)) != cudaSuccess)
        return bail(e, "upload");
    if ((e = cudaMemcpy(c->d_rope_lo, lo.data(), lo.size() * 4, cudaMemcpyHostToDevice)) != cudaSuccess)
        return bail(e, "upload");
    if ((e = cudaMemset(c->d_route_ctr, 0, bh * 4)) != cudaSuccess) return bail(e, "cudaMemset");
    if ((e = cudaMemset(c->d_err, 0, 4)) != cudaSuccess) return bail(e, "cudaMemset");

    *out = c;
    return HSQ_OK;
}

hsq_status hsq_destroy(hsq_ctx* ctx) {
    if (!ctx) return HSQ_OK;
    cudaDeviceSynchronize();
    free_ctx(ctx);
    return HSQ_OK;
}

hsq_status hsq_encode(hsq_ctx* ctx, const hsq_cache* cache, const void* K, const void* V,
                      hsq_dtype dtype, hsq_stream_t stream) {
    hsq_status st = check_common(ctx, cache);
    if (st != HSQ_OK) return st;
    if (!K || !V) return fail(ctx, HSQ_ERR_INVALID, "K or V is NULL");
    if (dtype != HSQ_DTYPE_F32 && dtype != HSQ_DTYPE_BF16) return fail(ctx, HSQ_ERR_INVALID, "bad dtype");
    cudaPointerAttributes pa;
    HSQ_CUDA(ctx, cudaPointerGetAttributes(&pa, cache->l3));
    const bool on_host = pa.type == cudaMemoryTypeHost;
    if (on_host != (cache->l3_on_host != 0))
        return fail(ctx, HSQ_ERR_INVALID, "l3 location does not match l3_on_host");
    if (on_host && pa.devicePointer != (void*)cache->l3)
        return fail(ctx, HSQ_ERR_INVALID, "host l3 is not mapped at the same address on the device");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    CacheView v = make_view(ctx, cache);
    l1_index_kernel<<<v.B, 1024, 0, s>>>(v, cache->l1_pos, cache->l1_count, ctx->d_prefix, ctx->d_err);
    EncodeOut o{cache->l1_kc, cache->l1_vc, cache->l1_kn, cache->l1_vn, cache->l2_kc, cache->l2_vc,
                cache->l2_kn, cache->l2_vn, cache->l2_cnt, cache->l3, ctx->d_prefix};
    dim3 grid(v.G, v.Hkv, v.B);
    const Tables tb = make_tables(ctx);
    if (v.N == 16) {
        if (dtype == HSQ_DTYPE_BF16) encode_kernel<16, true><<<grid, 16 * 32, 0, s>>>(v, o, K, V, tb);
        else encode_kernel<16, false><<<grid, 16 * 32, 0, s>>>(v, o, K, V, tb);
    } else {
        if (dtype == HSQ_DTYPE_BF16) encode_kernel<8, true><<<grid, 8 * 32, 0, s>>>(v, o, K, V, tb);
        else encode_kernel<8, false><<<grid, 8 * 32, 0, s>>>(v, o, K, V, tb);
    }
    return after_launch(ctx, "encode");
}

hsq_status hsq_route(hsq_ctx* ctx, const hsq_cache* cache, const float* q, const int32_t* pos,
                     int32_t* sel, float* scores_opt, hsq_stream_t stream) {
    hsq_status st = check_common(ctx, cache);
    if (st != HSQ_OK) return st;
    if (!q || !pos || !sel) return fail(ctx, HSQ_ERR_INVALID, "q, pos or sel is NULL");
    CacheView v = make_view(ctx, cache);
    RouteArgs a{q, pos, sel, scores_opt ? scores_opt : ctx->d_scores, ctx->d_route_ctr, ctx->d_err};
    st = dispatch_route(ctx, v, a, reinterpret_cast<cudaStream_t>(stream));
    if (st != HSQ_OK) return fail(ctx, st, "unsupported head ratio");
    return after_launch(ctx, "route");
}

hsq_status hsq_fetch_dequant(hsq_ctx* ctx, const hsq_cache* cache, const int32_t* sel,
                             float* k_out_opt, float* v_out_opt, uint8_t* valid_opt, hsq_stream_t stream) {
    hsq_status st = check_common(ctx, cache);
    if (st != HSQ_OK) return st;
    if (!sel) return fail(ctx, HSQ_ERR_INVALID, "sel is NULL");
    if (hsq::fault_mask() & HSQ_FAULT_FETCH) return fail(ctx, HSQ_ERR_CUDA, "injected fetch failure");
    CacheView v = make_view(ctx, cache);
    FetchArgs a{sel, k_out_opt, v_out_opt, valid_opt, cache->staging, ctx->d_err};
    dim3 grid(v.beta, v.B * v.Hkv);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (v.N == 16) fetch_kernel<16><<<grid, kThreads, 0, s>>>(v, a, make_tables(ctx));
    else fetch_kernel<8><<<grid, kThreads, 0, s>>>(v, a, make_tables(ctx));
    return after_launch(ctx, "fetch_dequant");
}

hsq_status hsq_decode_attn(hsq_ctx* ctx, const hsq_cache* cache, const float* q, const int32_t* pos,
                           const int32_t* sel, float* out, int flags, hsq_stream_t stream) {
    hsq_status st = check_common(ctx, cache);
    if (st != HSQ_OK) return st;
    if (!q || !pos || !sel || !out) return fail(ctx, HSQ_ERR_INVALID, "q, pos, sel or out is NULL");
    if (flags & ~HSQ_ATTN_FROM_STAGING) return fail(ctx, HSQ_ERR_INVALID, "unknown flags");
    const bool staged = (flags & HSQ_ATTN_FROM_STAGING) != 0;
    if (staged && !cache->staging) return fail(ctx, HSQ_ERR_INVALID, "staging is NULL");
    if (hsq::fault_mask() & HSQ_FAULT_FETCH) return fail(ctx, HSQ_ERR_CUDA, "injected fetch failure");
    const CacheView v = make_view(ctx, cache);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return dispatch_rn(ctx->r, v.N, [&](auto Ri, auto Ni) -> hsq_status {
        constexpr int R = decltype(Ri)::value, N = decltype(Ni)::value;
        const hsq_ctx::Plan p = decode_plan<R, N, false>(ctx, v.B, v.T);
        if (p.S == 0) return fail(ctx, HSQ_ERR_UNSUPPORTED, "decode kernel cannot be launched for this shape");
        DecodeArgs a{q, pos, const_cast<int32_t*>(sel), out, ctx->d_err, staged ? 1 : 0, 0};
        return launch_decode<R, N, false>(ctx, v, a, p, s);
    });
}

hsq_status hsq_decode_step(hsq_ctx* ctx, const hsq_cache* cache, const float* q, const int32_t* pos,
                           int32_t* sel, float* out, hsq_stream_t stream) {
    hsq_status st = check_common(ctx, cache);
    if (st != HSQ_OK) return st;
    if (!q || !pos || !sel || !out) return fail(ctx, HSQ_ERR_INVALID, "q, pos, sel or out is NULL");
    if (hsq::fault_mask() & HSQ_FAULT_FETCH) return fail(ctx, HSQ_ERR_CUDA, "injected fetch failure");
    const CacheView v = make_view(ctx, cache);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    bool fused = false;
    st = dispatch_rn(ctx->r, v.N, [&](auto Ri, auto Ni) -> hsq_status {
        constexpr int R = decltype(Ri)::value, N = decltype(Ni)::value;
        const hsq_ctx::Plan p = decode_plan<R, N, true>(ctx, v.B, v.T);
        if (p.S == 0) return HSQ_OK;  // no launchable cluster shape: two kernels below
        fused = true;
        DecodeArgs a{q, pos, sel, out, ctx->d_err, 0, 0};
        return launch_decode<R, N, true>(ctx, v, a, p, s);
    });
    if (st != HSQ_OK || fused) return st;
    st = hsq_route(ctx, cache, q, pos, sel, nullptr, stream);
    if (st != HSQ_OK) return st;
    return hsq_decode_attn(ctx, cache, q, pos, sel, out, 0, stream);
}

hsq_status hsq_sync_status(hsq_ctx* ctx, hsq_stream_t stream, int* device_word) {
    if (!ctx) return fail(nullptr, HSQ_ERR_INVALID, "context is NULL");
    HSQ_CUDA(ctx, cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)));
    int w = 0;
    HSQ_CUDA(ctx, cudaMemcpy(&w, ctx->d_err, 4, cudaMemcpyDeviceToHost));
    HSQ_CUDA(ctx, cudaMemset(ctx->d_err, 0, 4));
    if (device_word) *device_word = w;
    if (w) return fail(ctx, HSQ_ERR_DEVICE_CHECK, "device-side check failed (word " + std::to_string(w) + ")");
    return HSQ_OK;
}

const char* hsq_last_error(const hsq_ctx* ctx) {
    return ctx ? ctx->last_error.c_str() : hsq::process_error();
}

}  // extern "C"

// ===========================================================================
// Routing that allocates nothing.
//
// Some callers cannot call cudaMalloc: a serving runtime that reserves all
// device memory for its own pool at start-up and fails any later allocation,
// or a host that must not let a library call synchronise the device (a
// cudaMalloc may).  hsq_route_noalloc serves them.  It needs no context: the
// routing scores and the per-(b, h) tickets live in a fixed-size file-scope
// device array (every GPU that loads this library holds it until the process
// exits), the codebook in a small file-scope array filled once per device,
// and the query's RoPE angles are evaluated in float64 inside the kernel
// instead of being read from a context's tables.
// ===========================================================================

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[HSQ_NOALLOC_SCRATCH_BYTES];
static __device__ float g_noalloc_codebook[hsq::kCodebookFloats];

constexpr int kNoallocMaxDevices = 64;
std::mutex g_noalloc_mu;
unsigned char* g_noalloc_ptr[kNoallocMaxDevices] = {};

// Query RoPE from float64 angles p * theta^(-2i/d).
__device__ __forceinline__ void rope_f64(float v[8], int p, double theta) {
    const int l = hlane();
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int i = 4 * l + k;
        const double ang = (double)p * pow(theta, -2.0 * i / kDim);
        double sd, cd;
        sincos(ang, &sd, &cd);
        const float c = (float)cd, s = (float)sd;
        const float lo = v[k], hi = v[4 + k];
        v[k] = fmaf(lo, c, -hi * s);
        v[4 + k] = fmaf(hi, c, lo * s);
    }
}

template <int R>
__global__ void __launch_bounds__(kThreads) route_noalloc_kernel(CacheView c, RouteArgs a, double theta) {
    extern __shared__ uint32_t s_keys[];
    __shared__ float s_cb[hsq::kCodebookFloats];
    __shared__ float s_sign[kDim];
    __shared__ __align__(16) float s_q[R][kDim];
    __shared__ int s_hist[256];
    __shared__ int s_warp[32];
    __shared__ int s_flag;
    __shared__ uint32_t s_digit;
    __shared__ int s_above;

    const int bh = blockIdx.y, b = bh / c.Hkv, h = bh % c.Hkv;
    const int hw = threadIdx.x >> 4, l = hlane();
    const unsigned m = half_mask();
    for (int i = threadIdx.x; i < hsq::kCodebookFloats; i += blockDim.x) s_cb[i] = g_noalloc_codebook[i];
    for (int i = threadIdx.x; i < kDim; i += blockDim.x) s_sign[i] = (float)c.signs[i];
    __syncthreads();
    float sg[8];
    load_signs(sg, s_sign);

    if (hw < R) {
        const int j = h * R + hw;
        float x[8];
        load_f32x8(a.q + ((size_t)b * c.Hq + j) * kDim, x);
        rope_f64(x, __ldg(a.pos + b), theta);
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] *= sg[i];
        fwht(x, m);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            s_q[hw][4 * l + k] = x[k] * kRsqrtD;
            s_q[hw][64 + 4 * l + k] = x[4 + k] * kRsqrtD;
        }
    }
    __syncthreads();
    float gq[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int jj = 0; jj < R; ++jj) {
            s0 += s_q[jj][4 * l + k];
            s1 += s_q[jj][64 + 4 * l + k];
        }
        gq[k] = s0;
        gq[4 + k] = s1;
    }

    const int g_begin = blockIdx.x * kRouteGroupsPerCta;
    const int g_end = min(c.G, g_begin + kRouteGroupsPerCta);
    const float* c3 = s_cb + 32;
    for (int g = g_begin + hw; g < g_end; g += kHalves) {
        const int cnt = __ldg(c.l2_cnt + (size_t)b * c.G + g);
        float score = -INFINITY;
        if (cnt > 0) {
            const size_t go = (size_t)bh * c.G + g;
            float v[8];
            unpack3(reinterpret_cast<const uint32_t*>(c.l2_kc + go * 48), c3, 1.0f, v);
            float d = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) d = fmaf(gq[i], v[i], d);
            d = half_sum(d, m);
            score = __ldg(c.l2_kn + go) * d;
        }
        if (l == 0) a.scores[(size_t)bh * c.G + g] = score;
    }

    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const int ticket = atomicAdd(a.counters + bh, 1);
        s_flag = (ticket == (int)gridDim.x - 1);
    }
    __syncthreads();
    if (!s_flag) return;
    __threadfence();

    const int G = c.G, beta = c.beta;
    int ne_local = 0;
    for (int g = threadIdx.x; g < G; g += blockDim.x) {
        const uint32_t k = ordered_key(__ldcg(a.scores + (size_t)bh * G + g));
        s_keys[g] = k;
        ne_local += (k != 0u);
    }
    int ne;
    block_exclusive_scan(ne_local, s_warp, ne);

    uint32_t kstar = 0u;
    int need = 0;
    if (beta < ne) {
        uint32_t prefix = 0u, pmask = 0u;
        int remaining = beta;
        for (int shift = 24; shift >= 0; shift -= 8) {
            s_hist[threadIdx.x] = 0;
            __syncthreads();
            for (int g = threadIdx.x; g < G; g += blockDim.x) {
                const uint32_t k = s_keys[g];
                if ((k & pmask) == prefix) atomicAdd(&s_hist[(k >> shift) & 255u], 1);
            }
            __syncthreads();
            if (threadIdx.x < 32) {
                const int lane = threadIdx.x;
                int cnt[8], tot = 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) { cnt[i] = s_hist[255 - 8 * lane - i]; tot += cnt[i]; }
                int inc = tot;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    int y = __shfl_up_sync(0xffffffffu, inc, o);
                    if (lane >= o) inc += y;
                }
                const int exc = inc - tot;
                if (exc < remaining && inc >= remaining) {
                    int acc = exc;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        if (acc + cnt[i] >= remaining) {
                            s_digit = (uint32_t)(255 - 8 * lane - i);
                            s_above = acc;
                            break;
                        }
                        acc += cnt[i];
                    }
                }
            }
            __syncthreads();
            prefix |= s_digit << shift;
            pmask |= 255u << shift;
            remaining -= s_above;
            __syncthreads();
        }
        kstar = prefix;
        need = remaining;
    }

    const int per = (G + blockDim.x - 1) / blockDim.x;
    const int i0 = min(G, (int)threadIdx.x * per), i1 = min(G, i0 + per);
    int eq_local = 0;
    for (int g = i0; g < i1; ++g) eq_local += (s_keys[g] == kstar && kstar != 0u);
    int eq_total;
    const int eq_before = block_exclusive_scan(eq_local, s_warp, eq_total);
    int sel_local = 0;
    {
        int e = eq_before;
        for (int g = i0; g < i1; ++g) {
            const uint32_t k = s_keys[g];
            bool take = k > kstar;
            if (k == kstar && kstar != 0u) { take = e < need; ++e; }
            sel_local += take;
        }
    }
    int sel_total;
    int out = block_exclusive_scan(sel_local, s_warp, sel_total);
    {
        int e = eq_before;
        for (int g = i0; g < i1; ++g) {
            const uint32_t k = s_keys[g];
            bool take = k > kstar;
            if (k == kstar && kstar != 0u) { take = e < need; ++e; }
            if (take && out < beta) a.sel[(size_t)bh * beta + out++] = g;
        }
    }
    for (int i = sel_total + threadIdx.x; i < beta; i += blockDim.x) a.sel[(size_t)bh * beta + i] = -1;
    if (threadIdx.x == 0) a.counters[bh] = 0;
}

// One-time set-up of the current device: the scratch array's device address
// (a host-side use of the symbol name itself would not be a device address)
// and the codebook upload.  Synchronous, so it must not run under stream capture.
hsq_status noalloc_setup(unsigned char** scratch) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(nullptr, e, "cudaGetDevice");
    if (dev < 0 || dev >= kNoallocMaxDevices) return fail(nullptr, HSQ_ERR_UNSUPPORTED, "device ordinal above 63");
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_fail(nullptr, e, "cudaGetSymbolAddress(scratch)");
        float cb[hsq::kCodebookFloats];
        hsq::device_codebook(cb);
        e = cudaMemcpyToSymbol(g_noalloc_codebook, cb, sizeof(cb));
        if (e != cudaSuccess) return cuda_fail(nullptr, e, "cudaMemcpyToSymbol(codebook)");
        g_noalloc_ptr[dev] = static_cast<unsigned char*>(p);
    }
    *scratch = g_noalloc_ptr[dev];
    return HSQ_OK;
}

template <int R>
hsq_status launch_route_noalloc(const CacheView& v, const RouteArgs& a, double theta, cudaStream_t st, int dev) {
    const size_t smem = (size_t)v.G * 4;
    if (smem > 48 * 1024) {
        cudaError_t e = raise_smem_limit((const void*)route_noalloc_kernel<R>, dev, smem);
        if (e != cudaSuccess) return cuda_fail(nullptr, e, "cudaFuncSetAttribute");
    }
    dim3 grid((v.G + kRouteGroupsPerCta - 1) / kRouteGroupsPerCta, v.B * v.Hkv);
    route_noalloc_kernel<R><<<grid, kThreads, smem, st>>>(v, a, theta);
    return HSQ_OK;
}

}  // namespace

extern "C" hsq_status hsq_route_noalloc(const hsq_config* cfg, const hsq_cache* cache, const float* q,
                                        const int32_t* pos, int32_t* sel, hsq_stream_t stream) {
    std::string why = hsq::check_config(cfg);
    if (!why.empty()) return fail(nullptr, HSQ_ERR_INVALID, why);
    why = hsq::check_cache_shape(cfg, cache);
    if (!why.empty()) return fail(nullptr, HSQ_ERR_INVALID, why);
    if (!q || !pos || !sel) return fail(nullptr, HSQ_ERR_INVALID, "q, pos or sel is NULL");
    const int r = cfg->n_q_heads / cfg->n_kv_heads;
    if (!r_supported(r)) return fail(nullptr, HSQ_ERR_UNSUPPORTED, "r = Hq/Hkv must be 1, 2, 4, 5 or 8");
    const size_t bh = (size_t)cache->B * cfg->n_kv_heads;
    const size_t G = (size_t)hsq::groups_of(cache->T, cfg->group_n);
    const size_t ticket_bytes = (bh * 4 + 255) / 256 * 256;
    if (ticket_bytes + bh * G * 4 > (size_t)HSQ_NOALLOC_SCRATCH_BYTES)
        return fail(nullptr, HSQ_ERR_INVALID,
                    "B * n_kv_heads * ceil(T / group_n) too large for the fixed 4 MiB scratch of hsq_route_noalloc");
    if (G * 4 > 200 * 1024) return fail(nullptr, HSQ_ERR_INVALID, "ceil(T / group_n) above 51200");
    unsigned char* scratch = nullptr;
    hsq_status st = noalloc_setup(&scratch);
    if (st != HSQ_OK) return st;
    int dev = 0;
    cudaGetDevice(&dev);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // the tickets must start at zero on every call (the array keeps the last call's contents)
    cudaError_t e = cudaMemsetAsync(scratch, 0, ticket_bytes, s);
    if (e != cudaSuccess) return cuda_fail(nullptr, e, "cudaMemsetAsync(tickets)");
    CacheView v{};
    v.B = cache->B; v.T = cache->T; v.N = cfg->group_n; v.G = (int)G;
    v.Hkv = cfg->n_kv_heads; v.Hq = cfg->n_q_heads; v.beta = cfg->beta;
    v.max_l1 = cfg->max_l1; v.W = hsq::bitmap_words(cache->T);
    v.l2_kc = cache->l2_kc; v.l2_kn = cache->l2_kn; v.l2_cnt = cache->l2_cnt; v.signs = cache->signs;
    RouteArgs a{q, pos, sel, reinterpret_cast<float*>(scratch + ticket_bytes),
                reinterpret_cast<int*>(scratch), nullptr};
    switch (r) {
        case 1: st = launch_route_noalloc<1>(v, a, cfg->rope_theta, s, dev); break;
        case 2: st = launch_route_noalloc<2>(v, a, cfg->rope_theta, s, dev); break;
        case 4: st = launch_route_noalloc<4>(v, a, cfg->rope_theta, s, dev); break;
        case 5: st = launch_route_noalloc<5>(v, a, cfg->rope_theta, s, dev); break;
        default: st = launch_route_noalloc<8>(v, a, cfg->rope_theta, s, dev); break;
    }
    if (st != HSQ_OK) return st;
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(nullptr, e, "route_noalloc");
    return HSQ_OK;
}
