// Device-side building blocks shared by the HSQ kernels (included by every
// translation unit that holds kernels; each gets its own internal copy).
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
// A half-warp is the unit of work; where both halves of a warp run the same
// code with warp-uniform loop bounds the shuffles use the full-warp mask.
//
// All arithmetic is fp32.  Softmax runs in the log2 domain (logits scaled by
// log2(e)/sqrt(128), exp2).
#pragma once

#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "hsq_ctx.h"

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
    int cap;  // tokens the layout is sized for (G = ceil(cap / N) groups, W = ceil(cap / 32) words)
    int rot;  // 1: TurboQuant rotation Pi; 0: Plain-KV (identity, signs NULL)
    // Heads: the view has Hkv selection heads (per-(b, h) selections, scores,
    // staging, CTAs); view head h reads the tiers of buffer head h / hdiv of
    // Hb.  hdiv = 1, Hb = Hkv except under per-query-head routing, where the
    // view heads are the query heads (Hkv = Hq, hdiv = Hq / Hb).
    int hdiv, Hb;
    // TQ-QKV key-residual sketches (NULL unless cfg.qjl)
    const float* qjl_s; const uint32_t* l1_qs; const float* l1_qn; const uint32_t* l3_qs; const float* l3_qn;
    const uint8_t* l1_kc; const uint8_t* l1_vc; const float* l1_kn; const float* l1_vn;
    const int32_t* l1_pos; const int32_t* l1_count;
    const uint8_t* l2_kc; const uint8_t* l2_vc; const float* l2_kn; const float* l2_vn;
    const uint8_t* l2_cnt;
    const uint8_t* l3;
    const uint32_t* l1_bitmap;
    const int8_t* signs;
    const uint8_t* staging;
    // hot-group table (fused decode step; NULL without one): slot i of view head bh
    // at hot_rec + (bh * (hot_mask + 1) + i) * N * 136, its group in hot_tag
    uint8_t* hot_rec;
    int32_t* hot_tag;
    int hot_mask;  // slots - 1
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

// Full-warp mask for shuffles of code that every warp runs converged (both
// half-warps together, loop bounds uniform across the warp).
constexpr unsigned kFull = 0xffffffffu;

// Lane l of a half-warp holds, after spread_sum<K>, the sum of value
// spread_index<K>(l): the first log2(K) halving steps (offsets 8, 4, 2, 1)
// each keep half of the values per lane, so K values cost K - 1 shuffles
// instead of 4 K.
template <int K>
__device__ __forceinline__ int spread_index(int l) {
    int idx = 0;
    if (K >= 2) idx += ((l >> 3) & 1) * (K / 2);
    if (K >= 4) idx += ((l >> 2) & 1) * (K / 4);
    if (K >= 8) idx += ((l >> 1) & 1) * (K / 8);
    if (K >= 16) idx += (l & 1) * (K / 16);
    return idx;
}

template <int M>
__device__ __forceinline__ void spread_halve(float* v, int off, bool up) {
#pragma unroll
    for (int i = 0; i < M / 2; ++i) {
        const float send = up ? v[i] : v[i + M / 2];
        const float keep = up ? v[i + M / 2] : v[i];
        v[i] = keep + __shfl_xor_sync(kFull, send, off, 16);
    }
}

// Sums each of v[0..K) over the 16 lanes of the half-warp (K a power of two
// up to 16; v is overwritten).  Returns the sum of v[spread_index<K>(lane)].
template <int K>
__device__ __forceinline__ float spread_sum(float (&v)[K]) {
    static_assert(K == 1 || K == 2 || K == 4 || K == 8 || K == 16, "K must be a power of two <= 16");
    const int l = hlane();
    if constexpr (K >= 2) spread_halve<K>(v, 8, l & 8);
    if constexpr (K >= 4) spread_halve<K / 2>(v, 4, l & 4);
    if constexpr (K >= 8) spread_halve<K / 4>(v, 2, l & 2);
    if constexpr (K >= 16) spread_halve<K / 8>(v, 1, l & 1);
    float s = v[0];
    if constexpr (K < 16) s += __shfl_xor_sync(kFull, s, 1, 16);
    if constexpr (K < 8) s += __shfl_xor_sync(kFull, s, 2, 16);
    if constexpr (K < 4) s += __shfl_xor_sync(kFull, s, 4, 16);
    if constexpr (K < 2) s += __shfl_xor_sync(kFull, s, 8, 16);
    return s;
}

__host__ __device__ constexpr int pow2_ceil(int x) { return x <= 1 ? 1 : 2 * pow2_ceil((x + 1) / 2); }

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
// The two table rows RoPE at position p combines (p = 256 a + c: cos/sin of
// 256 a omega and of c omega, this lane's 4 frequencies), loaded ahead of use.
struct RopeRows {
    float4 ch, sh, cl, sl;
};

__device__ __forceinline__ RopeRows rope_rows(int p, const Tables& tb) {
    const int l = hlane();
    const float* rh = tb.rope_hi + (size_t)(p >> 8) * kDim;
    const float* rl = tb.rope_lo + (size_t)(p & 255) * kDim;
    RopeRows r;
    r.ch = __ldg(reinterpret_cast<const float4*>(rh + 4 * l));
    r.sh = __ldg(reinterpret_cast<const float4*>(rh + 64 + 4 * l));
    r.cl = __ldg(reinterpret_cast<const float4*>(rl + 4 * l));
    r.sl = __ldg(reinterpret_cast<const float4*>(rl + 64 + 4 * l));
    return r;
}

// Rotate-half RoPE of this lane's dims (i, i + 64), the angle by addition:
// cos(A + B) = cA cB - sA sB, sin(A + B) = sA cB + cA sB.
__device__ __forceinline__ void rope_apply(float v[8], const RopeRows& r) {
    const float cA[4] = {r.ch.x, r.ch.y, r.ch.z, r.ch.w}, sA[4] = {r.sh.x, r.sh.y, r.sh.z, r.sh.w};
    const float cB[4] = {r.cl.x, r.cl.y, r.cl.z, r.cl.w}, sB[4] = {r.sl.x, r.sl.y, r.sl.z, r.sl.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float c = fmaf(cA[k], cB[k], -sA[k] * sB[k]);
        const float s = fmaf(sA[k], cB[k], cA[k] * sB[k]);
        const float lo = v[k], hi = v[4 + k];
        v[k] = fmaf(lo, c, -hi * s);
        v[4 + k] = fmaf(hi, c, lo * s);
    }
}

__device__ __forceinline__ void rope(float v[8], int p, const Tables& tb) { rope_apply(v, rope_rows(p, tb)); }

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

// Codec forward: y = Pi (x / n) with Pi = H diag(s) / sqrt(d) (TurboQuant),
// or y = x / n (Plain-KV, rot false).  Returns n.
__device__ __forceinline__ float tq_rotate(float x[8], float y[8], const float sg[8], unsigned m, bool rot) {
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) ss = fmaf(x[i], x[i], ss);
    ss = half_sum(ss, m);
    const float n = sqrtf(ss);
    const float inv = n > 0.f ? 1.0f / n : 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) y[i] = x[i] * inv;
    if (rot) {
#pragma unroll
        for (int i = 0; i < 8; ++i) y[i] *= sg[i];
        fwht(y, m);
#pragma unroll
        for (int i = 0; i < 8; ++i) y[i] *= kRsqrtD;
    }
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

// The same through L2 only (ld.global.cg): for caller buffers that may be
// page-locked host memory read in place over the host link.
__device__ __forceinline__ void load_f32x8_cg(const float* p, float v[8]) {
    const int l = hlane();
    const float4 a = __ldcg(reinterpret_cast<const float4*>(p + 4 * l));
    const float4 b = __ldcg(reinterpret_cast<const float4*>(p + 64 + 4 * l));
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
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
    for (int i = threadIdx.x; i < kDim; i += blockDim.x) s_sign[i] = signs ? (float)signs[i] : 1.f;
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
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
// wait until at most n committed groups of this thread are still in flight
template <int n>
__device__ __forceinline__ void cp_async_wait_group() { asm volatile("cp.async.wait_group %0;\n" ::"n"(n) : "memory"); }

// bytes: a multiple of 16, both addresses 16-byte aligned
__device__ __forceinline__ void stage16(void* dst, const void* src, int bytes) {
    uint8_t* d = static_cast<uint8_t*>(dst);
    const uint8_t* s = static_cast<const uint8_t*>(src);
#pragma unroll 1
    for (int i = threadIdx.x * 16; i < bytes; i += blockDim.x * 16) cp_async16(d + i, s + i);
}

__device__ __forceinline__ void stage4(float* dst, const float* src, int n) {
#pragma unroll 1
    for (int i = threadIdx.x; i < n; i += blockDim.x) cp_async4(dst + i, src + i);
}

// signs of the lane's 8 dims straight from global memory (all +1 without signs)
__device__ __forceinline__ void load_signs_global(float s[8], const int8_t* __restrict__ signs) {
    const int l = hlane();
    if (!signs) {
#pragma unroll
        for (int i = 0; i < 8; ++i) s[i] = 1.f;
        return;
    }
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
    int agg_max;  // score = max over the query heads instead of their sum
};

__device__ __forceinline__ uint32_t ordered_key(float s) {
    if (s == -INFINITY) return 0u;
    const uint32_t u = __float_as_uint(s + 0.0f);  // -0 and +0 are one score (one key)
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_to_float(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

constexpr int kSelBins = 2048;          // histogram bins of the bucket select (8 per thread)
constexpr int kSelMaxGroups = 32768;
constexpr int kSelCand = 32;            // boundary candidates ranked by one warp

struct __align__(16) SelectSmem {
    int hist[kSelBins + 4];  // + a sink bin for keys out of play (branch-free histogram)
    uint32_t taken[kSelMaxGroups / 32];
    uint32_t cand_key[kSelCand];
    int cand_g[kSelCand];
    uint32_t red[3][32];  // per warp (up to 32 warps)
    int wsum[32];
    int bstar, above, bcnt, ncand;
};

// Block-wide exclusive scan of one int per thread (NT threads) with a single
// barrier.  `wsum` must not be written again before the block's next __syncthreads.
template <int NT>
__device__ __forceinline__ int block_scan_1(int v, int* wsum, int& total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFull, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    int before = 0, t = 0;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) {
        const int s = wsum[w];
        before += w < warp ? s : 0;
        t += s;
    }
    total = t;
    return before + x - v;
}

// Top-beta selection by the whole block (NT threads, a multiple of 32, at
// least 256).  s_keys[0..G) are
// order-preserving keys of the fp32 group scores (0 = empty group, never
// selected).  The groups of the beta largest keys (ties to the lower group)
// go to out[0..beta) in ascending group order, -1 padded (out may be shared
// or global memory; the caller synchronises before reading it).  stats, when
// not null, holds nstats partial (count, max, min) statistics of the
// non-empty keys (4 words each) that together cover all G keys; otherwise
// they are computed here.
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
//
// Layout: warp w owns the contiguous keys [w W, (w + 1) W), W = 32 kpw;
// step j of a warp reads keys w W + 32 j + lane (conflict-free), and the
// ordered placement counts with one ballot per step.  Every loop bound is
// uniform, so all warp-level operations are converged, and the per-key work
// is branch-free (clamped loads, bitwise flags, a sink bin): a divergent
// branch around a load or an atomic costs several hundred cycles per step.
template <int NT>
__device__ void select_top_beta(const uint32_t* s_keys, int G, int beta, int* out, SelectSmem& ss,
                                const uint32_t* stats = nullptr, int nstats = 0) {
    static_assert(NT % 32 == 0 && NT >= kSelBins / 8, "block size");
    constexpr int NW = NT / 32;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int kpw = (G + NT - 1) / NT;  // steps per warp
    const int wbase = warp * 32 * kpw;
    auto key_at = [&](int j, int& i) -> uint32_t {
        i = wbase + 32 * j + lane;
        const uint32_t v = s_keys[min(i, G - 1)];
        return i < G ? v : 0u;
    };

    // count, max and min of the non-empty keys
    int ne = 0;
    uint32_t lo = 0xFFFFFFFFu, hi = 0u;
    if (stats) {
#pragma unroll 1
        for (int w = tid; w < (G + 31) / 32; w += NT) ss.taken[w] = 0u;
#pragma unroll 1
        for (int r = 0; r < nstats; ++r) {
            ne += (int)stats[4 * r];
            hi = max(hi, stats[4 * r + 1]);
            lo = min(lo, stats[4 * r + 2]);
        }
        __syncthreads();
    } else {
        int cn = 0;
        uint32_t mx = 0u, mn = 0xFFFFFFFFu;
#pragma unroll 1
        for (int j = 0; j < kpw; ++j) {
            int i;
            const uint32_t v = key_at(j, i);
            cn += v != 0u;
            mx = max(mx, v);
            mn = min(mn, v != 0u ? v : 0xFFFFFFFFu);
        }
        cn = __reduce_add_sync(kFull, cn);
        mx = __reduce_max_sync(kFull, mx);
        mn = __reduce_min_sync(kFull, mn);
        if (lane == 0) { ss.red[0][warp] = (uint32_t)cn; ss.red[1][warp] = mx; ss.red[2][warp] = mn; }
#pragma unroll 1
        for (int w = tid; w < (G + 31) / 32; w += NT) ss.taken[w] = 0u;
        __syncthreads();
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            ne += (int)ss.red[0][w];
            hi = max(hi, ss.red[1][w]);
            lo = min(lo, ss.red[2][w]);
        }
    }

    // mode 0: take every non-empty group; 1: keys > bhi plus the ranked
    // boundary candidates; 2: keys > kstar plus the first `need` equal to kstar
    int mode = 0, above = 0, need = 0, mode1_base = 0;
    uint32_t bhi = 0u, kstar = 0u;
    if (ne > beta) {
        const float smin = key_to_float(lo), smax = key_to_float(hi);
        const float fscale = (float)kSelBins / (smax - smin);
        const bool float_ok = isfinite(fscale) && smax > smin;
#pragma unroll 1
        for (int level = 0; level < 8; ++level) {
            if (lo == hi) { mode = 2; kstar = lo; need = beta - above; break; }
            const bool fl = level == 0 && float_ok;
            const int bits = 32 - __clz(hi - lo);
            const int shift = bits > 11 ? bits - 11 : 0;
            auto bin_of = [&](uint32_t v) -> int {
                if (fl) return min(max((int)((key_to_float(v) - smin) * fscale), 0), kSelBins - 1);
                return (int)((v - lo) >> shift);
            };
            for (int q = tid; q < kSelBins / 4; q += NT) reinterpret_cast<int4*>(ss.hist)[q] = make_int4(0, 0, 0, 0);
            __syncthreads();
#pragma unroll 1
            for (int j = 0; j < kpw; ++j) {
                int i;
                const uint32_t v = key_at(j, i);
                const bool play = (v != 0u) & (v >= lo) & (v <= hi);
                atomicAdd(&ss.hist[play ? bin_of(v) : kSelBins], 1);
            }
            __syncthreads();
            // blocked scan from the top: thread t < B/8 owns bins [B - 8(t+1), B - 8t)
            const bool owns = tid < kSelBins / 8;
            const int top = kSelBins - 8 * min(tid, kSelBins / 8 - 1);
            const int4 h0 = *reinterpret_cast<const int4*>(&ss.hist[top - 8]);
            const int4 h1 = *reinterpret_cast<const int4*>(&ss.hist[top - 4]);
            int hv[8] = {h1.w, h1.z, h1.y, h1.x, h0.w, h0.z, h0.y, h0.x};  // descending bins
            int local = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                hv[i] = owns ? hv[i] : 0;
                local += hv[i];
            }
            int tot;
            int run = above + block_scan_1<NT>(local, ss.wsum, tot);
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
            // the boundary bin's members: gathered (when few) and their exact key
            // range; and per warp the keys above the boundary bin (all taken)
            uint32_t bmx = 0u, bmn = 0xFFFFFFFFu;
            int wsure = 0;
#pragma unroll 1
            for (int j = 0; j < kpw; ++j) {
                int i;
                const uint32_t v = key_at(j, i);
                const bool inr = (v != 0u) & (v >= lo) & (v <= hi);
                const int bn = bin_of(v);
                const bool inb = inr & (bn == bstar);
                wsure += __popc(__ballot_sync(kFull, (v > hi) | (inr & (bn > bstar))));
                bmx = max(bmx, inb ? v : 0u);
                bmn = min(bmn, inb ? v : 0xFFFFFFFFu);
                const unsigned bm = __ballot_sync(kFull, inb);
                if (bm != 0u && bcnt <= kSelCand) {  // rare: the boundary bin's few keys
                    int slot = 0;
                    if (lane == 0) slot = atomicAdd(&ss.ncand, __popc(bm));
                    slot = __shfl_sync(kFull, slot, 0) + __popc(bm & ((1u << lane) - 1u));
                    if (inb) {
                        ss.cand_key[slot] = v;
                        ss.cand_g[slot] = i;
                    }
                }
            }
            bmx = __reduce_max_sync(kFull, bmx);
            bmn = __reduce_min_sync(kFull, bmn);
            if (lane == 0) { ss.red[0][warp] = (uint32_t)wsure; ss.red[1][warp] = bmx; ss.red[2][warp] = bmn; }
            __syncthreads();
            uint32_t blo_b = 0xFFFFFFFFu, bhi_b = 0u;
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                bhi_b = max(bhi_b, ss.red[1][w]);
                blo_b = min(blo_b, ss.red[2][w]);
            }
            if (bcnt <= kSelCand) {
                // every warp ranks the candidates (same result); warp 0 records the taken ones
                const uint32_t ck = lane < bcnt ? ss.cand_key[lane] : 0u;
                const int cg = lane < bcnt ? ss.cand_g[lane] : -1;
                int rank = 0;
#pragma unroll 1
                for (int j = 0; j < bcnt; ++j) {
                    const uint32_t kj = __shfl_sync(kFull, ck, j);
                    const int gj = __shfl_sync(kFull, cg, j);
                    rank += (kj > ck) || (kj == ck && gj < cg);
                }
                const bool tk = lane < bcnt && rank < need;
                if (warp == 0 && tk) atomicOr(&ss.taken[cg >> 5], 1u << (cg & 31));
                // where this warp's taken keys start: keys above the bin plus taken
                // candidates, over the warps before it (the placement needs no count pass)
                const int ow = cg >= 0 ? cg / (32 * kpw) : -1;
                int base = 0;
#pragma unroll
                for (int w = 0; w < NW; ++w) {
                    const int cw = (int)ss.red[0][w] + __popc(__ballot_sync(kFull, tk & (ow == w)));
                    base += w < warp ? cw : 0;
                }
                mode1_base = base;
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

    // ordered placement: per step a ballot of taken (mode 2: greater) and of
    // equal keys; a warp's counts, then one exclusive scan over the warps
    // (mode is uniform; the per-key expressions are bitwise, without branches)
    const uint32_t thr = mode == 0 ? 0u : mode == 1 ? bhi : kstar;
    auto flags_at = [&](int j, int& i, bool& gt, bool& eq) {
        const uint32_t v = key_at(j, i);
        const uint32_t tw = ss.taken[min(i, G - 1) >> 5];
        const bool tk = (mode == 1) & (v != 0u) & (((tw >> (i & 31)) & 1u) != 0u);
        gt = (v > thr) | tk;
        eq = (mode == 2) & (v == kstar);
    };
    int pos_gt = mode1_base, eq_before = 0;
    if (mode != 1) {
        int wgt = 0, weq = 0;
#pragma unroll 1
        for (int j = 0; j < kpw; ++j) {
            int i;
            bool gt, eq;
            flags_at(j, i, gt, eq);
            wgt += __popc(__ballot_sync(kFull, gt));
            weq += __popc(__ballot_sync(kFull, eq));
        }
        int total;
        const int packed = block_scan_1<NT>(lane == 0 ? (wgt | (weq << 16)) : 0, ss.wsum, total);
        pos_gt = __shfl_sync(kFull, packed, 0) & 0xFFFF;
        eq_before = __shfl_sync(kFull, packed, 0) >> 16;
    }
    const unsigned lt = (1u << lane) - 1u;
#pragma unroll 1
    for (int j = 0; j < kpw; ++j) {
        int i;
        bool gt, eq;
        flags_at(j, i, gt, eq);
        const unsigned bg = __ballot_sync(kFull, gt), be = __ballot_sync(kFull, eq);
        const int pg = pos_gt + __popc(bg & lt), pe = eq_before + __popc(be & lt);
        const int p = gt ? pg + (mode == 2 ? min(pe, need) : 0) : pg + pe;
        const bool put = (gt | (eq & (pe < need))) & (p < beta);
        if (put) out[p] = i;
        pos_gt += __popc(bg);
        eq_before += __popc(be);
    }
    const int n_sel = mode == 0 ? ne : beta;
#pragma unroll 1
    for (int i = n_sel + tid; i < beta; i += NT) out[i] = -1;
}

// Dot products of two 128-vectors (a, b; this lane's 8 dims each) with the R
// query heads.  Returns the lane's share of the 2R sums (spread_sum): index
// idx < R is head idx of a, R <= idx < 2R head idx - R of b, idx >= 2R unused.
template <int R>
__device__ __forceinline__ float pair_dots(const float (&q)[R][8], const float (&ka)[8], const float (&kb)[8],
                                           int& idx) {
    constexpr int K = pow2_ceil(2 * R);
    float p[K];
#pragma unroll
    for (int j = 0; j < R; ++j) {
        float da = 0.f, db = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            da = fmaf(q[j][k], ka[k], da);
            db = fmaf(q[j][k], kb[k], db);
        }
        p[j] = da;
        p[R + j] = db;
    }
#pragma unroll
    for (int j = 2 * R; j < K; ++j) p[j] = 0.f;
    idx = spread_index<K>(hlane());
    return spread_sum<K>(p);
}

// pair_dots of (q, ka, kb) plus (q2, ka2, kb2) in one reduction: the lane
// products of both are summed before the spread.
template <int R>
__device__ __forceinline__ float pair_dots2(const float (&q)[R][8], const float (&ka)[8], const float (&kb)[8],
                                            const float (&q2)[R][8], const float (&ka2)[8], const float (&kb2)[8],
                                            int& idx) {
    constexpr int K = pow2_ceil(2 * R);
    float p[K];
#pragma unroll
    for (int j = 0; j < R; ++j) {
        float da = 0.f, db = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            da = fmaf(q[j][k], ka[k], da);
            db = fmaf(q[j][k], kb[k], db);
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            da = fmaf(q2[j][k], ka2[k], da);
            db = fmaf(q2[j][k], kb2[k], db);
        }
        p[j] = da;
        p[R + j] = db;
    }
#pragma unroll
    for (int j = 2 * R; j < K; ++j) p[j] = 0.f;
    idx = spread_index<K>(hlane());
    return spread_sum<K>(p);
}

// Routing scores of two groups a and b: (sum_j q~_j) . c3[codes], every lane
// gets both.  One fixed summation order, shared by the routing kernel and
// the decode step, so both select the same groups.
__device__ __forceinline__ void route_pair(const float (&gq)[8], const float (&va)[8], const float (&vb)[8],
                                           float& sa, float& sb) {
    float p[2] = {0.f, 0.f};
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        p[0] = fmaf(gq[k], va[k], p[0]);
        p[1] = fmaf(gq[k], vb[k], p[1]);
    }
    const float s = spread_sum<2>(p);
    sa = __shfl_sync(kFull, s, 0, 16);
    sb = __shfl_sync(kFull, s, 8, 16);
}

// Rotated, RoPE'd query heads of KV head h: every half-warp computes head
// min(hw, R - 1) (all warps stay converged); half-warps hw < R store it.
// x: that head's query (this lane's 8 dims).  With qr, the RoPE'd query in
// the original frame is stored too.  rot false (Plain-KV): no rotation.
template <int R>
__device__ __forceinline__ void prepare_queries(float (&x)[8], int pos, const float sg[8], const Tables& tb,
                                                float (*s_qt)[kDim], float (*s_qr)[kDim], bool rot) {
    const int hw = threadIdx.x >> 4, l = hlane();
    const int j = min(hw, R - 1);
    rope(x, pos, tb);
    if (s_qr && hw < R) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            s_qr[j][4 * l + k] = x[k];
            s_qr[j][64 + 4 * l + k] = x[4 + k];
        }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] *= sg[i];
    if (rot) fwht(x, kFull);
    const float sc = rot ? kRsqrtD : 1.f;
    if (hw < R) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            s_qt[j][4 * l + k] = x[k] * sc;
            s_qt[j][64 + 4 * l + k] = x[4 + k] * sc;
        }
    }
}

// The same, loading the query heads (q: the KV head's first query head).
template <int R>
__device__ __forceinline__ void prepare_queries(const float* __restrict__ q, int pos, const float sg[8],
                                                const Tables& tb, float (*s_qt)[kDim], float (*s_qr)[kDim],
                                                bool rot) {
    float x[8];  // (only the R half-warps of the heads read; the rest compute on zeros)
    if ((int)threadIdx.x >> 4 < R) {
        load_f32x8_cg(q + (size_t)(threadIdx.x >> 4) * kDim, x);
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] = 0.f;
    }
    prepare_queries<R>(x, pos, sg, tb, s_qt, s_qr, rot);
}

__host__ __device__ inline unsigned al16(size_t x) { return (unsigned)((x + 15) & ~(size_t)15); }

__host__ __device__ inline unsigned route_smem_bytes(int G) {
    return al16((size_t)G * 4) + kRouteGroupsPerCta * (48 + 4 + 1);
}

// ---------------------------------------------------------------------------
// Selection validity: entries must be -1 or in [0, G), non-negative entries
// strictly ascending and before any -1.
// ---------------------------------------------------------------------------

__device__ __forceinline__ int valid_sel(const int32_t* __restrict__ row, int i, int G, int* err) {
    const int g = __ldcg(row + i);
    if (g < 0) return -1;
    bool ok = g < G;
    if (i > 0) {
        const int p = __ldcg(row + i - 1);
        ok = ok && p >= 0 && p < g;
    }
    if (!ok) {
        atomicOr(err, HSQ_DEVERR_SEL);
        return -1;
    }
    return g;
}


// Kernel-side views of a context and a cache (host helpers).
inline CacheView make_view(const hsq_ctx* ctx, const hsq_cache* c) {
    CacheView v{};
    // layout strides follow the capacity; groups and bitmap words past T are empty
    const int cap = c->t_cap > 0 ? c->t_cap : c->T;
    v.B = c->B; v.T = c->T; v.N = ctx->cfg.group_n; v.G = hsq::groups_of(cap, v.N);
    v.Hkv = ctx->cfg.n_kv_heads; v.Hq = ctx->cfg.n_q_heads; v.beta = ctx->cfg.beta;
    v.max_l1 = ctx->cfg.max_l1; v.W = hsq::bitmap_words(cap); v.cap = cap;
    v.l1_kc = c->l1_kc; v.l1_vc = c->l1_vc; v.l1_kn = c->l1_kn; v.l1_vn = c->l1_vn;
    v.l1_pos = c->l1_pos; v.l1_count = c->l1_count;
    v.l2_kc = c->l2_kc; v.l2_vc = c->l2_vc; v.l2_kn = c->l2_kn; v.l2_vn = c->l2_vn; v.l2_cnt = c->l2_cnt;
    v.l3 = c->l3; v.l1_bitmap = c->l1_bitmap; v.staging = c->staging;
    v.rot = ctx->cfg.codec == HSQ_CODEC_PLAIN ? 0 : 1;
    v.signs = v.rot ? c->signs : nullptr;
    v.hdiv = 1; v.Hb = v.Hkv;
    if (ctx->cfg.qjl) {
        v.qjl_s = c->qjl_s; v.l1_qs = c->l1_qs; v.l1_qn = c->l1_qn; v.l3_qs = c->l3_qs; v.l3_qn = c->l3_qn;
    }
    if (ctx->cfg.hot_slots > 0) {
        v.hot_rec = c->hot_rec; v.hot_tag = c->hot_tag; v.hot_mask = ctx->cfg.hot_slots - 1;
    }
    return v;
}

// The view the routing, fetch and decode kernels run on: one selection per
// KV head, or per query head under per-query-head routing.
inline CacheView make_sel_view(const hsq_ctx* ctx, const hsq_cache* c) {
    CacheView v = make_view(ctx, c);
    if (ctx->cfg.route_per_head) {
        v.hdiv = v.Hq / v.Hkv;
        v.Hkv = v.Hq;
    }
    return v;
}

// sqrt(pi/2) / m for the m = 128-bit residual sketch: E[sign(s . rho) (s . q)] =
// sqrt(2/pi) (q . rho) / |rho| for s ~ N(0, I).
constexpr float kQjlScale = 0.0097915167f;

// This lane's 8 sketch signs times w (coordinates 4l + k and 64 + 4l + k of
// the 128-bit sketch in words wd): +w where the bit is set, else -w.
__device__ __forceinline__ void sketch_signs(uint4 wd, float w, float s[8]) {
    const int l = hlane();
    const uint32_t lo = ((l >> 3) ? wd.y : wd.x) >> (4 * (l & 7));
    const uint32_t hi = ((l >> 3) ? wd.w : wd.z) >> (4 * (l & 7));
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        s[k] = ((lo >> k) & 1u) ? w : -w;
        s[4 + k] = ((hi >> k) & 1u) ? w : -w;
    }
}

// Row of the tier buffers that view head (b, h) reads.
__device__ __forceinline__ size_t buf_head(const CacheView& c, int b, int h) {
    return (size_t)b * c.Hb + h / c.hdiv;
}

inline Tables make_tables(const hsq_ctx* ctx) {
    Tables t{};
    t.cb = ctx->d_cb; t.rope_hi = ctx->d_rope_hi; t.rope_lo = ctx->d_rope_lo; t.max_pos = ctx->cfg.max_pos;
    return t;
}

}  // namespace
