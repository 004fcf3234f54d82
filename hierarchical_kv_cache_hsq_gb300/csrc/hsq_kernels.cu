// HSQ kernels for GB300 (sm_103a) other than the decode step (encode,
// routing, fetch), the routing-only entry point that allocates nothing, and
// the C entry points.  The decode-step kernel lives in hsq_decode.cuh and is
// compiled per head ratio in hsq_decode_r*.cu.
//
// Method: Tamarin (HSQ) technical summary (gist.science rs-10297225),
// section 2; TurboQuant: "Ablation, Statistical Inference, and Validation
// for KV-Cache Compression" (gist.science 2607.09683), experimental setup
// item 1.

#include <cooperative_groups.h>
#include <cuda.h>  // driver types only (CUcontext, CUresult): entry points are looked up at run time
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <algorithm>
#include <mutex>
#include <type_traits>
#include <string>
#include <vector>

#include "hsq_ctx.h"
#include "hsq_device.cuh"
#include "hsq_tc.cuh"

namespace {

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
    auto word = [&](int w) -> uint32_t {  // bits at t >= T (up to the capacity) do not count
        uint32_t x = c.l1_bitmap[(size_t)b * W + w];
        const int valid = c.T - 32 * w;
        if (valid < 32) x = valid <= 0 ? 0u : x & ((1u << valid) - 1u);
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
    float* win_kv; float* gsum; int recent;  // growth state (win_kv NULL: none)
    // prefill: the attention's key (RoPE'd, bf16 hi + lo) and transposed value
    // operand images, 64-key tiles (hsq_prefill.cu); used by the kPF variant only
    uint8_t* pf_kh; uint8_t* pf_kl; uint8_t* pf_vt; int pf_nkt;
    // TQ-QKV: a device copy of every L3 record's key codes and norms,
    // [B][Hkv][G][N * 64 | N * 4] (NULL: none)
    uint8_t* kc3;
};

// TQ3 of one group summary (this half-warp's 8 dims of the mean; x is
// overwritten) into its 48-byte code row and its norm.  w: this half's 12
// shared words, zero on entry; the whole warp is converged (both halves call it).
__device__ __forceinline__ void write_summary(float x[8], const float sg[8], unsigned m, bool rot, const float* t3,
                                              uint32_t* w, uint8_t* codes, float* norm) {
    const int l = hlane();
    float ys[8];
    const float ns = tq_rotate(x, ys, sg, m, rot);
    uint32_t fa = 0, fb = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        fa |= (uint32_t)quant3(ys[k], t3) << (3 * k);
        fb |= (uint32_t)quant3(ys[4 + k], t3) << (3 * k);
    }
    const int bit = 12 * l, wi = bit >> 5, sh = bit & 31;
    atomicOr(&w[wi], fa << sh);
    if (sh > 20) atomicOr(&w[wi + 1], fa >> (32 - sh));
    atomicOr(&w[6 + wi], fb << sh);
    if (sh > 20) atomicOr(&w[6 + wi + 1], fb >> (32 - sh));
    __syncwarp();
    if (l < 12) reinterpret_cast<uint32_t*>(codes)[l] = w[l];
    if (l == 0) *norm = ns;
}

// (48 resident warps per SM -- 3 CTAs of 16 warps or 6 of 8, 40 registers: the
// kernel is issue bound and the extra warps hide its memory and shared-memory
// latencies; 32 warps measured 20 % slower.)  A CTA takes kEncGroups
// consecutive groups: each warp encodes its token of every group in turn, then
// warp j forms group j's summary, so the summaries run side by side.
constexpr int kEncGroups = 4;
// dynamic shared memory of the encode kernel: the member rows s_sum[kEncGroups][N][2][128]
constexpr size_t enc_dyn_smem(int N) { return (size_t)kEncGroups * N * 2 * 128 * 4; }
// kRot: TurboQuant rotation (false: Plain-KV), fixed at compile time
// kPF: prefill, the same encode also writes the attention's K/V operand images
template <int N, bool kBF16, bool kRot, bool kPF = false>
__global__ void __launch_bounds__(N * 32, 16 * 3 / N) encode_kernel(CacheView c, EncodeOut o, const void* __restrict__ Kp,
                                                        const void* __restrict__ Vp, Tables tb) {
    __shared__ float s_cb[hsq::kCodebookFloats];
    __shared__ float s_sign[kDim];
    __shared__ __align__(16) uint8_t s_rec[kEncGroups][N * 136];
    extern __shared__ __align__(16) float s_dyn_enc[];
    auto s_sum = reinterpret_cast<float (*)[N][2][kDim]>(s_dyn_enc);  // [kEncGroups][N][2][128]
    __shared__ int s_member[kEncGroups][N];
    __shared__ uint32_t s_l2[kEncGroups][2][12];

    const int h = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, half = (threadIdx.x >> 4) & 1, l = hlane();
    const unsigned m = half_mask();
    load_tables(s_cb, s_sign, tb, c.signs);
    if (threadIdx.x < kEncGroups * 24) (&s_l2[0][0][0])[threadIdx.x] = 0u;
    __syncthreads();
    const float* t4 = s_cb + 16;
    const float* t3 = s_cb + 40;
    float sg[8];
    load_signs(sg, s_sign);

#pragma unroll 1
    for (int j = 0; j < kEncGroups; ++j) {  // token `warp` of each of the CTA's groups
        const int g = blockIdx.x * kEncGroups + j;
        if (g >= c.G) break;
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

        // the recent window's inputs, for decode-time growth (slot t mod recent)
        if (o.win_kv && in_ctx && t >= c.T - o.recent) {
            float* wp = o.win_kv + ((((size_t)b * c.Hkv + h) * o.recent + t % o.recent) * 2 + half) * kDim;
            *reinterpret_cast<float4*>(wp + 4 * l) = make_float4(x[0], x[1], x[2], x[3]);
            *reinterpret_cast<float4*>(wp + 64 + 4 * l) = make_float4(x[4], x[5], x[6], x[7]);
        }

        // L3: TQ4 of the raw (pre-RoPE) key / value
        float y[8];
        const float n = tq_rotate(x, y, sg, m, kRot);
        uint16_t lo, hi;
        pack4(y, t4, lo, hi);
        {
            uint8_t* row = s_rec[j] + (half ? N * 64 : 0) + warp * 64;
            reinterpret_cast<uint16_t*>(row)[l] = lo;
            reinterpret_cast<uint16_t*>(row + 32)[l] = hi;
            if (l == 0) reinterpret_cast<float*>(s_rec[j] + N * 128)[half * N + warp] = n;
        }

        // RoPE'd key (half 0) for L1 and for the group summary; values as they are
        float xr[8];
    #pragma unroll
        for (int i = 0; i < 8; ++i) xr[i] = x[i];
        if (half == 0 && in_ctx) rope(xr, t, tb);

        if (kPF && t < o.pf_nkt * 64) {  // row t & 63 of key tile t >> 6 (zero past T)
            const int row = t & 63;
            const size_t img = (((size_t)b * c.Hkv + h) * o.pf_nkt + (t >> 6)) * (64 * kDim * 2);
            if (half == 0) {
    #pragma unroll
                for (int blk = 0; blk < 2; ++blk) {
                    uint16_t hi[4], lo[4];
    #pragma unroll
                    for (int k = 0; k < 4; ++k) hsq_tc::split_bf16(xr[4 * blk + k], hi[k], lo[k]);
                    const uint32_t off = hsq_tc::sw128_row_quad(64, row, blk, l);
                    *reinterpret_cast<uint2*>(o.pf_kh + img + off) =
                        make_uint2((uint32_t)hi[0] | ((uint32_t)hi[1] << 16), (uint32_t)hi[2] | ((uint32_t)hi[3] << 16));
                    *reinterpret_cast<uint2*>(o.pf_kl + img + off) =
                        make_uint2((uint32_t)lo[0] | ((uint32_t)lo[1] << 16), (uint32_t)lo[2] | ((uint32_t)lo[3] << 16));
                }
            } else {
    #pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int d = (i < 4 ? 4 * l : 64 + 4 * l) + (i & 3);
                    *reinterpret_cast<uint16_t*>(o.pf_vt + img + hsq_tc::sw128_elem(d, row)) =
                        __bfloat16_as_ushort(__float2bfloat16_rn(x[i]));
                }
            }
        }

        if (is_l1 && slot < c.max_l1) {
            const size_t so = ((size_t)b * c.Hkv + h) * c.max_l1 + slot;
            if (half == 0) {
                float yr[8];
                tq_rotate(xr, yr, sg, m, kRot);  // same norm as the raw key (RoPE is norm preserving)
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
            float* row = &s_sum[j][warp][half][0];
            *reinterpret_cast<float4*>(row + 4 * l) = make_float4(xr[0], xr[1], xr[2], xr[3]);
            *reinterpret_cast<float4*>(row + 64 + 4 * l) = make_float4(xr[4], xr[5], xr[6], xr[7]);
        }
        if (threadIdx.x == warp * 32) s_member[j][warp] = member ? 1 : 0;
    }
    __syncthreads();

    // L3 records out (16-byte chunks; through the host link when L3 is pinned host memory)
    {
        const int g0 = blockIdx.x * kEncGroups;
        const int ng = min(kEncGroups, c.G - g0);
        uint4* dst = reinterpret_cast<uint4*>(o.l3 + (((size_t)b * c.Hkv + h) * c.G + g0) * (N * 136));
        const uint4* src = reinterpret_cast<const uint4*>(&s_rec[0][0]);
        for (int i = threadIdx.x; i < ng * (N * 136 / 16); i += blockDim.x) dst[i] = src[i];
        if (o.kc3) {  // the key codes (chunks 0 .. 4N) and key norms (chunks 8N .. 8N + N/4) again
            constexpr int kKC = N * 68 / 16;
            uint4* kd = reinterpret_cast<uint4*>(o.kc3 + (((size_t)b * c.Hkv + h) * c.G + g0) * (N * 68));
            for (int i = threadIdx.x; i < ng * kKC; i += blockDim.x) {
                const int j = i / kKC, r = i - j * kKC;
                kd[i] = src[j * (N * 136 / 16) + (r < 4 * N ? r : 4 * N + r)];
            }
        }
    }

    // L2 summaries, group j by warp j: mean over members in token order, then TQ3
    const int j = warp, g = blockIdx.x * kEncGroups + warp;
    if (j < kEncGroups && g < c.G) {
        int cnt = 0;
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.f;
        for (int k = 0; k < N; ++k) {
            if (!s_member[j][k]) continue;
            ++cnt;
            const float* row = &s_sum[j][k][half][0];
            const float4 a = *reinterpret_cast<const float4*>(row + 4 * l);
            const float4 bq = *reinterpret_cast<const float4*>(row + 64 + 4 * l);
            acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
            acc[4] += bq.x; acc[5] += bq.y; acc[6] += bq.z; acc[7] += bq.w;
        }
        // growth: the running sums of the group holding position T - recent
        // (its members below that position; zero when no token has left yet)
        const int p_next = c.T - o.recent;
        if (o.win_kv && (p_next >= 0 ? g == p_next / N : g == 0)) {
            float* gs = o.gsum + ((size_t)b * c.Hkv + h) * hsq::kGsumFloats;
            const bool keep = p_next >= 0;
            *reinterpret_cast<float4*>(gs + half * kDim + 4 * l) =
                keep ? make_float4(acc[0], acc[1], acc[2], acc[3]) : make_float4(0.f, 0.f, 0.f, 0.f);
            *reinterpret_cast<float4*>(gs + half * kDim + 64 + 4 * l) =
                keep ? make_float4(acc[4], acc[5], acc[6], acc[7]) : make_float4(0.f, 0.f, 0.f, 0.f);
            if ((threadIdx.x & 31) == 0) {
                gs[2 * kDim] = keep ? (float)cnt : 0.f;
                gs[2 * kDim + 1] = (float)p_next;  // the window's first position at encode
            }
        }
        if (cnt > 0) {
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = acc[i] / (float)cnt;
        }
        const size_t go = ((size_t)b * c.Hkv + h) * c.G + g;
        write_summary(acc, sg, m, kRot, t3, s_l2[j][half], (half ? o.l2_vc : o.l2_kc) + go * 48,
                      (half ? o.l2_vn : o.l2_kn) + go);
        if ((threadIdx.x & 31) == 0 && h == 0) o.l2_cnt[(size_t)b * c.G + g] = (uint8_t)cnt;
    }
}

// ---------------------------------------------------------------------------
// TQ-QKV, encode side: the 1-bit sketches of the key residuals, one half-warp
// per residual (qjl_kernel: L3, qjl_l1_kernel: L1).  The sketch of a residual rho taken in the rotated frame is sign(S Pi rho');
// with rho' the residual in the original frame, S Pi is one fixed matrix per
// layer, so the kernel forms rho' and multiplies by S Pi (formed once per
// encode, `qjl_pack_kernel`):
//   L3: rho' = RoPE(k_t - k^_t, t),  k^_t = n Pi^T c^ (c^: the stored codes'
//       codebook values, n: the stored norm);
//   L1: rho' = RoPE(k_t, t) - n Pi^T c^1 (c^1: the stored L1 codes).
// Both read the codes encode_kernel wrote (the L3 key codes from a device
// copy, the L1 codes from the tier), so the residual is that of the stored
// codes by construction; one inverse transform per residual.
// ---------------------------------------------------------------------------

struct SketchOut {
    // S Pi as the B operand of the m16n8k16 tensor-core product (k = dimension d,
    // n = sketch row i), in fragment order: for n-tile nt (rows 8 nt ..) and
    // k-step ks (dims 16 ks ..), lane (g, q) = (lane / 4, lane % 4) holds at
    // [(nt * 8 + ks) * 32 + lane] the bf16 pairs {M[i][d], M[i][d + 1]} and
    // {M[i][d + 8], M[i][d + 9]}, M = S Pi, i = 8 nt + g, d = 16 ks + 2 q, of
    // M's bf16 rounding (hi) and of the bf16 rounding of the remainder (lo)
    const uint4* Sf; uint32_t* l1_qs; float* l1_qn; uint32_t* l3_qs; float* l3_qn;
    const uint8_t* kc3;  // the L3 key codes and norms, [B][Hkv][G][N * 64 | N * 4]
};

__device__ __forceinline__ void split_pair(float a, float b, uint32_t& hi, uint32_t& lo) {
    const __nv_bfloat16 ha = __float2bfloat16_rn(a), hb = __float2bfloat16_rn(b);
    const __nv_bfloat16 la = __float2bfloat16_rn(a - __bfloat162float(ha));
    const __nv_bfloat16 lb = __float2bfloat16_rn(b - __bfloat162float(hb));
    hi = (uint32_t)__bfloat16_as_ushort(ha) | ((uint32_t)__bfloat16_as_ushort(hb) << 16);
    lo = (uint32_t)__bfloat16_as_ushort(la) | ((uint32_t)__bfloat16_as_ushort(lb) << 16);
}

// M = S Pi = S H diag(s) / sqrt(d): row i of M is s / sqrt(d) times the
// Hadamard transform of row i of S (H is symmetric); M = S without rotation.
// One CTA per n-tile (8 rows), one warp per row (4 dims per lane), then the
// tile's 256 fragments.
__global__ void __launch_bounds__(256) qjl_pack_kernel(const float* __restrict__ S, const int8_t* __restrict__ signs,
                                                       int rot, uint4* __restrict__ Sf) {
    __shared__ float s_m[8][kDim + 4];
    const int nt = blockIdx.x, w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float4 v = __ldg(reinterpret_cast<const float4*>(S + (size_t)(8 * nt + w) * kDim) + lane);
    if (rot) {
        float a[4] = {v.x + v.y, v.x - v.y, v.z + v.w, v.z - v.w};  // index bit 0
        float t[4] = {a[0] + a[2], a[1] + a[3], a[0] - a[2], a[1] - a[3]};  // index bit 1
#pragma unroll
        for (int sft = 1; sft < 32; sft <<= 1) {  // index bits 2..6 = lane bits 0..4
            const float sgn = (lane & sft) ? -1.f : 1.f;
#pragma unroll
            for (int k = 0; k < 4; ++k) t[k] = fmaf(sgn, t[k], __shfl_xor_sync(kFull, t[k], sft));
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) t[k] *= (float)__ldg(signs + 4 * lane + k) * kRsqrtD;
        v = make_float4(t[0], t[1], t[2], t[3]);
    }
    *reinterpret_cast<float4*>(&s_m[w][4 * lane]) = v;
    __syncthreads();
    const int ks = threadIdx.x >> 5, gq = lane >> 2, d = 16 * ks + 2 * (lane & 3);
    const float* row = &s_m[gq][d];
    uint4 f;
    split_pair(row[0], row[1], f.x, f.z);
    split_pair(row[8], row[9], f.y, f.w);
    Sf[(nt * 8 + ks) * 32 + lane] = f;
}

// Four 8 x 8 b16 matrices from shared memory (ldmatrix.x4): lanes 8 j .. 8 j + 7
// give the row addresses of matrix j; register j holds this lane's pair of it.
__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// D += A B for one m16n8k16 tile: bf16 operands, fp32 accumulators
__device__ __forceinline__ void mma_bf16_16816(float d[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// bits 0..3 of x to bits 0, 2, 4, 6
__device__ __forceinline__ uint32_t spread4(uint32_t x) {
    return (x & 1u) | ((x & 2u) << 1) | ((x & 4u) << 2) | ((x & 8u) << 3);
}

// Residual rows of the sketch pass, the A operand of M rho': [row][bf16 pairs],
// kQRS words per row (4 words of pad: the fragment loads hit distinct banks).
constexpr int kQRS = kDim / 2 + 4;
constexpr int kQjlThreads = 256;  // 8 warps: warp w takes sketch rows 16 w .. 16 w + 15

// This half-warp's 8 dims of one residual into its hi / lo operand rows; returns |rho'|.
__device__ __forceinline__ float qjl_row(const float rho[8], uint32_t* rh, uint32_t* rl, unsigned m) {
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) ss = fmaf(rho[i], rho[i], ss);
    const int l = hlane();
    uint2 h0, l0, h1, l1;
    split_pair(rho[0], rho[1], h0.x, l0.x);
    split_pair(rho[2], rho[3], h0.y, l0.y);
    split_pair(rho[4], rho[5], h1.x, l1.x);
    split_pair(rho[6], rho[7], h1.y, l1.y);
    *reinterpret_cast<uint2*>(rh + 2 * l) = h0;  // dims 4 l .. 4 l + 3
    *reinterpret_cast<uint2*>(rl + 2 * l) = l0;
    *reinterpret_cast<uint2*>(rh + 32 + 2 * l) = h1;  // dims 64 + 4 l ..
    *reinterpret_cast<uint2*>(rl + 32 + 2 * l) = l1;
    return sqrtf(half_sum(ss, m));
}

// D[r][i] = sum_d rho'_r[d] M[i][d] for kM 16-row tiles of residual rows on the
// tensor cores, operands split into bf16 hi + lo and the three products hi hi,
// hi lo, lo hi accumulated in fp32 (about 2^-16 relative per term); bit i of row
// r's sketch (word i / 32, bit i % 32) is set in s_bits[r] (zero on entry) when
// D >= 0.  Each B fragment is loaded once for the kM tiles.
template <int kM>
__device__ __forceinline__ void qjl_products(const uint32_t (*rh)[kQRS], const uint32_t (*rl)[kQRS],
                                             const uint4* __restrict__ Sf, uint32_t (*s_bits)[4]) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gq = lane >> 2, tq = lane & 3;
    float d[kM][2][4];
#pragma unroll
    for (int mt = 0; mt < kM; ++mt)
#pragma unroll
        for (int j = 0; j < 2; ++j) d[mt][j][0] = d[mt][j][1] = d[mt][j][2] = d[mt][j][3] = 0.f;
    // ldmatrix.x4 row addresses: lane L gives row (L & 7) + 8 ((L >> 3) & 1) of the
    // tile and the 8-dim half (L >> 4) of the k-step: matrices 0..3 are the A
    // fragment's a0..a3 (rows 0-7 / 8-15, dims 0-7 / 8-15 of the 16 x 16 block)
    const int lrow = (lane & 7) + 8 * ((lane >> 3) & 1), lcol = 4 * (lane >> 4);
    const uint32_t rh0 = (uint32_t)__cvta_generic_to_shared(&rh[lrow][lcol]);
    const uint32_t rl0 = (uint32_t)__cvta_generic_to_shared(&rl[lrow][lcol]);
#pragma unroll 2
    for (int ks = 0; ks < 8; ++ks) {
        const uint4 bf0 = __ldg(Sf + ((2 * warp) * 8 + ks) * 32 + lane);
        const uint4 bf1 = __ldg(Sf + ((2 * warp + 1) * 8 + ks) * 32 + lane);
#pragma unroll
        for (int mt = 0; mt < kM; ++mt) {
            const uint32_t off = (uint32_t)((16 * mt * kQRS + 8 * ks) * 4);
            uint32_t ah0, ah1, ah2, ah3, al0, al1, al2, al3;
            ldmatrix_x4(rh0 + off, ah0, ah1, ah2, ah3);
            ldmatrix_x4(rl0 + off, al0, al1, al2, al3);
            mma_bf16_16816(d[mt][0], al0, al1, al2, al3, bf0.x, bf0.y);  // lo hi
            mma_bf16_16816(d[mt][0], ah0, ah1, ah2, ah3, bf0.z, bf0.w);  // hi lo
            mma_bf16_16816(d[mt][0], ah0, ah1, ah2, ah3, bf0.x, bf0.y);  // hi hi
            mma_bf16_16816(d[mt][1], al0, al1, al2, al3, bf1.x, bf1.y);
            mma_bf16_16816(d[mt][1], ah0, ah1, ah2, ah3, bf1.z, bf1.w);
            mma_bf16_16816(d[mt][1], ah0, ah1, ah2, ah3, bf1.x, bf1.y);
        }
    }
#pragma unroll
    for (int mt = 0; mt < kM; ++mt) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {  // D[g][2q + c], D[g + 8][2q + c] -> bytes of rows g, g + 8
            const int nt = 2 * warp + j;
            const uint32_t b0 = __ballot_sync(kFull, d[mt][j][0] >= 0.f), b1 = __ballot_sync(kFull, d[mt][j][1] >= 0.f);
            const uint32_t b2 = __ballot_sync(kFull, d[mt][j][2] >= 0.f), b3 = __ballot_sync(kFull, d[mt][j][3] >= 0.f);
            if (tq == 0) {
                const uint32_t lo = spread4((b0 >> (4 * gq)) & 15u) | (spread4((b1 >> (4 * gq)) & 15u) << 1);
                const uint32_t hi = spread4((b2 >> (4 * gq)) & 15u) | (spread4((b3 >> (4 * gq)) & 15u) << 1);
                atomicOr(&s_bits[16 * mt + gq][nt >> 2], lo << (8 * (nt & 3)));
                atomicOr(&s_bits[16 * mt + gq + 8][nt >> 2], hi << (8 * (nt & 3)));
            }
        }
    }
}

// The L3 sketches: 64 consecutive tokens of one (sequence b, KV head h) per CTA,
// four per half-warp.  Token t's residual is rho' = RoPE(k_t - n Pi^T c^, t), c^ and n
// its stored L3 codes' codebook values and norm.
constexpr int kQjlTok = 64;

template <int N, bool kBF16>
__global__ void __launch_bounds__(kQjlThreads, 4) qjl_kernel(CacheView c, SketchOut o, const void* __restrict__ Kp,
                                                            Tables tb) {
    __shared__ float s_cb[hsq::kCodebookFloats];
    __shared__ float s_sign[kDim];
    __shared__ __align__(16) uint32_t s_rh[kQjlTok][kQRS], s_rl[kQjlTok][kQRS];
    __shared__ uint32_t s_bits[kQjlTok][4];

    const int h = blockIdx.y, b = blockIdx.z, hw = threadIdx.x >> 4, l = hlane();
    const unsigned m = half_mask();
    const int t0 = blockIdx.x * kQjlTok;
    const size_t bh = (size_t)b * c.Hkv + h;
    load_tables(s_cb, s_sign, tb, c.signs);
    (&s_bits[0][0])[threadIdx.x] = 0u;  // kQjlTok * 4 == kQjlThreads
    __syncthreads();
    const float* c4 = s_cb;
    float sg[8];
    load_signs(sg, s_sign);
#pragma unroll 2
    for (int i = 0; i < kQjlTok / 16; ++i) {
        const int r = hw + 16 * i, t = t0 + r;
        const bool valid = t < c.T;  // rows past the context: zero
        const int tc = valid ? t : c.T - 1;
        const int g = tc / N, k = tc - g * N;
        const uint8_t* kr = o.kc3 + (bh * c.G + g) * (N * 68);
        const uint32_t lo = *reinterpret_cast<const uint16_t*>(kr + k * 64 + 2 * l);
        const uint32_t hi = *reinterpret_cast<const uint16_t*>(kr + k * 64 + 32 + 2 * l);
        const float n = *reinterpret_cast<const float*>(kr + N * 64 + 4 * k);
        float x[8];
        const size_t off = (bh * c.T + tc) * kDim;
        if (kBF16) load_bf16x8(static_cast<const uint16_t*>(Kp) + off, x);
        else load_f32x8(static_cast<const float*>(Kp) + off, x);
        const RopeRows rr = rope_rows(tc, tb);
        float rho[8];  // k^ = n Pi^T c^ = diag(s) H (n / sqrt(d) c^)
        unpack4(lo, hi, c4, n * kRsqrtD, rho);
        fwht(rho, m);
#pragma unroll
        for (int j = 0; j < 8; ++j) rho[j] = valid ? x[j] - sg[j] * rho[j] : 0.f;
        rope_apply(rho, rr);
        const float gamma = qjl_row(rho, s_rh[r], s_rl[r], m);
        if (valid && l == 0) o.l3_qn[bh * c.G * N + t] = gamma;
    }
    __syncthreads();
    qjl_products<kQjlTok / 16>(s_rh, s_rl, o.Sf, s_bits);
    __syncthreads();
    const int r = threadIdx.x >> 2;
    if (t0 + r < c.T) o.l3_qs[(bh * c.G * N + t0 + r) * 4 + (threadIdx.x & 3)] = s_bits[r][threadIdx.x & 3];
}

// The L1 sketches: 16 L1 slots of one (b, h) per CTA, one per half-warp.  Slot e
// holds position p = l1_pos[b][e]; its residual is rho' = RoPE(k_p, p) - n Pi^T c^1,
// c^1 its stored L1 codes' codebook values and n its stored norm.
template <bool kBF16>
__global__ void __launch_bounds__(kQjlThreads) qjl_l1_kernel(CacheView c, SketchOut o, const void* __restrict__ Kp,
                                                           Tables tb) {
    __shared__ float s_cb[hsq::kCodebookFloats];
    __shared__ float s_sign[kDim];
    __shared__ __align__(16) uint32_t s_rh[16][kQRS], s_rl[16][kQRS];
    __shared__ uint32_t s_bits[16][4];

    const int h = blockIdx.y, b = blockIdx.z, hw = threadIdx.x >> 4, l = hlane();
    const unsigned m = half_mask();
    const int cnt = min(c.l1_count[b], c.max_l1);
    const int e0 = blockIdx.x * 16;
    if (e0 >= cnt) return;  // (uniform over the CTA, before any barrier)
    const size_t bh = (size_t)b * c.Hkv + h;
    load_tables(s_cb, s_sign, tb, c.signs);
    if (threadIdx.x < 64) (&s_bits[0][0])[threadIdx.x] = 0u;
    __syncthreads();
    const float* c4 = s_cb;
    float sg[8];
    load_signs(sg, s_sign);
    const int e = e0 + hw;
    const bool valid = e < cnt;
    const int ec = valid ? e : cnt - 1;
    const int p = c.l1_pos[(size_t)b * c.max_l1 + ec];
    const size_t so = bh * c.max_l1 + ec;
    const uint32_t lo = *reinterpret_cast<const uint16_t*>(c.l1_kc + so * 64 + 2 * l);
    const uint32_t hi = *reinterpret_cast<const uint16_t*>(c.l1_kc + so * 64 + 32 + 2 * l);
    const float n = c.l1_kn[so];
    float x[8];
    const size_t off = (bh * c.T + p) * kDim;
    if (kBF16) load_bf16x8(static_cast<const uint16_t*>(Kp) + off, x);
    else load_f32x8(static_cast<const float*>(Kp) + off, x);
    rope(x, p, tb);
    float rho[8];
    unpack4(lo, hi, c4, n * kRsqrtD, rho);
    fwht(rho, m);
#pragma unroll
    for (int j = 0; j < 8; ++j) rho[j] = valid ? x[j] - sg[j] * rho[j] : 0.f;
    const float gamma = qjl_row(rho, s_rh[hw], s_rl[hw], m);
    if (valid && l == 0) o.l1_qn[bh * c.max_l1 + e] = gamma;
    __syncthreads();
    qjl_products<1>(s_rh, s_rl, o.Sf, s_bits);
    __syncthreads();
    if (threadIdx.x < 64 && e0 + (threadIdx.x >> 2) < cnt)
        o.l1_qs[(bh * c.max_l1 + e0 + (threadIdx.x >> 2)) * 4 + (threadIdx.x & 3)] = s_bits[threadIdx.x >> 2][threadIdx.x & 3];
}

// ---------------------------------------------------------------------------
// Decode-time growth: append one token per sequence at position T.  One CTA
// per sequence b: warp h < Hkv for KV head h (half 0 the key, half 1 the
// value), and one more warp (warp 0 when there are 32 KV heads) for the
// sequence's L1 bookkeeping: the L1 slot of the new token -- the slot of the
// token p = T - recent that leaves the window, or a new slot when nothing
// leaves -- and the sequence's L1 list, count and bitmap (no other CTA touches
// them).  While that warp searches, the head warps write the new token's L3
// record slot and, when p leaves (p >= sinks), add p's input (from the window
// ring) to the running sums of its group in position order and re-quantise
// the group's summary, as the encode of the longer context computes it; once
// the slot is known they write the L1 entry.  (A p >= sinks that is not in L1
// cannot happen in a cache built by hsq_encode and hsq_append; the search
// flags it, HSQ_DEVERR_GROW.)
// ---------------------------------------------------------------------------

template <int N, bool kBF16>
__global__ void __launch_bounds__(1024) append_kernel(CacheView c, EncodeOut o, int32_t* l1_pos, int32_t* l1_count,
                                                      uint32_t* l1_bitmap, const void* __restrict__ kp,
                                                      const void* __restrict__ vp, Tables tb, int sinks,
                                                      int recent, int* err) {
    __shared__ float s_cb[hsq::kCodebookFloats];
    __shared__ float s_sign[kDim];
    __shared__ uint32_t s_l2[32][2][12];
    __shared__ int s_slot;
    const int b = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int keeper = c.Hkv < 32 ? c.Hkv : 0;  // the bookkeeping warp
    const bool head = warp < c.Hkv;
    const int h = head ? warp : 0;
    const int half = (threadIdx.x >> 4) & 1, l = hlane();
    const unsigned m = half_mask();
    const int t = c.T, p = t - recent;
    const bool leaves = p >= 0 && p >= sinks;  // p leaves the window (a sink stays)
    const size_t bh = (size_t)b * c.Hkv + h;
    // loads that depend on nothing, issued first
    float x[8];
    if (kBF16) load_bf16x8(static_cast<const uint16_t*>(half ? vp : kp) + bh * kDim, x);
    else load_f32x8(static_cast<const float*>(half ? vp : kp) + bh * kDim, x);
    float* wp = o.win_kv + ((bh * recent + (size_t)(t % recent)) * 2 + half) * kDim;  // = p's ring slot
    float xp[8];
    load_f32x8_cg(wp, xp);
    // the RoPE rows of t and p and the running sums, none waiting on the slot
    const RopeRows rope_t = rope_rows(t, tb), rope_p = rope_rows(max(p, 0), tb);
    const float* gs0 = o.gsum + bh * hsq::kGsumFloats;
    const float4 gs_a = __ldcg(reinterpret_cast<const float4*>(gs0 + half * kDim + 4 * l));
    const float4 gs_b = __ldcg(reinterpret_cast<const float4*>(gs0 + half * kDim + 64 + 4 * l));
    const float gs_n = __ldcg(gs0 + 2 * kDim);
    load_tables(s_cb, s_sign, tb, c.signs);
    if (threadIdx.x < 24 * c.Hkv) (&s_l2[0][0][0])[threadIdx.x] = 0u;

    auto bookkeeping = [&]() {  // the slot, and the sequence's L1 bookkeeping
        int32_t* pos = l1_pos + (size_t)b * c.max_l1;
        const int cnt = min(__ldcg(l1_count + b), c.max_l1);
        int slot = -1, found_p = 0;
        if (leaves) {
            // the window fills the last `recent` slots, rotated: the token at
            // position x0 + j (x0 its first position at encode) is in slot
            // cnt - recent + j mod recent -- checked, else every slot is scanned
            const int x0 = (int)__ldcg(o.gsum + (size_t)b * c.Hkv * hsq::kGsumFloats + 2 * kDim + 1);
            const int pred = x0 >= 0 && p >= x0 && cnt >= recent ? cnt - recent + (p - x0) % recent : -1;
            int found = pred >= 0 && __ldcg(pos + pred) == p ? pred : -1;
            if (found < 0) {
                int f = -1;
#pragma unroll 4
                for (int i = lane; i < cnt; i += 32)  // independent loads, no early exit
                    f = __ldcg(pos + i) == p ? i : f;
                found = __reduce_max_sync(kFull, f);
            }
            if (found >= 0) {
                slot = found;
                found_p = 1;
            } else if (lane == 0) {
                atomicOr(err, HSQ_DEVERR_GROW);
            }
        } else if (cnt < c.max_l1) {
            slot = cnt;
            if (lane == 0) l1_count[b] = cnt + 1;
        } else if (lane == 0) {
            atomicOr(err, HSQ_DEVERR_L1_OVER);
        }
        if (lane == 0) {
            uint32_t* bm = l1_bitmap + (size_t)b * c.W;
            if (slot >= 0) {
                pos[slot] = t;
                atomicOr(bm + (t >> 5), 1u << (t & 31));
            }
            if (found_p) atomicAnd(bm + (p >> 5), ~(1u << (p & 31)));
            s_slot = slot;
        }
    };
    __syncthreads();  // the tables are in shared memory
    // (a warp of its own runs beside the heads; with 32 KV heads warp 0 does both)
    if (warp == keeper) bookkeeping();
    const float* t4 = s_cb + 16;
    const float* t3 = s_cb + 40;
    float sg[8];
    load_signs(sg, s_sign);

    float n = 0.f;
    uint16_t lo = 0, hi = 0;
    if (head) {
        // L3 record slot t: TQ4 of the raw key / value
        float y[8];
        n = tq_rotate(x, y, sg, m, c.rot);
        pack4(y, t4, lo, hi);
        uint8_t* rec = o.l3 + (bh * c.G + t / N) * (N * 136);
        uint8_t* row = rec + (half ? N * 64 : 0) + (t % N) * 64;
        reinterpret_cast<uint16_t*>(row)[l] = lo;
        reinterpret_cast<uint16_t*>(row + 32)[l] = hi;
        if (l == 0) reinterpret_cast<float*>(rec + N * 128)[half * N + t % N] = n;
        if (c.hot_tag && lane == 0) {  // the hot-group table's copy of group t / N is stale
            int32_t* tag = c.hot_tag + bh * (c.hot_mask + 1) + ((t / N) & c.hot_mask);
            if (*tag == t / N) *tag = -1;
        }
        if (leaves) {
            if (half == 0) rope_apply(xp, rope_p);
            float* gs = o.gsum + bh * hsq::kGsumFloats;
            const bool fresh = p % N == 0;  // p opens its group: nothing summed before it
            float acc[8];
            const float4 a = fresh ? make_float4(0.f, 0.f, 0.f, 0.f) : gs_a;
            const float4 bq = fresh ? make_float4(0.f, 0.f, 0.f, 0.f) : gs_b;
            acc[0] = a.x + xp[0]; acc[1] = a.y + xp[1]; acc[2] = a.z + xp[2]; acc[3] = a.w + xp[3];
            acc[4] = bq.x + xp[4]; acc[5] = bq.y + xp[5]; acc[6] = bq.z + xp[6]; acc[7] = bq.w + xp[7];
            const int cnt = (fresh ? 0 : (int)gs_n) + 1;
            __syncwarp();  // every lane has read the count before lane 0 rewrites it
            *reinterpret_cast<float4*>(gs + half * kDim + 4 * l) = make_float4(acc[0], acc[1], acc[2], acc[3]);
            *reinterpret_cast<float4*>(gs + half * kDim + 64 + 4 * l) = make_float4(acc[4], acc[5], acc[6], acc[7]);
            if (lane == 0) gs[2 * kDim] = (float)cnt;
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = acc[i] / (float)cnt;
            const int gp = p / N;
            const size_t go = bh * c.G + gp;
            write_summary(acc, sg, m, c.rot, t3, s_l2[h][half], (half ? o.l2_vc : o.l2_kc) + go * 48,
                          (half ? o.l2_vn : o.l2_kn) + go);
            if (lane == 0 && h == 0) o.l2_cnt[(size_t)b * c.G + gp] = (uint8_t)cnt;
        }
        // t's inputs replace p's in the ring (p's were read at the start)
        *reinterpret_cast<float4*>(wp + 4 * l) = make_float4(x[0], x[1], x[2], x[3]);
        *reinterpret_cast<float4*>(wp + 64 + 4 * l) = make_float4(x[4], x[5], x[6], x[7]);
    }
    __syncthreads();  // the slot is known
    const int slot = s_slot;
    // L1 entry (RoPE'd key, value as coded for L3)
    if (head && slot >= 0) {
        const size_t so = bh * c.max_l1 + slot;
        if (half == 0) {
            float xr[8], yr[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) xr[i] = x[i];
            rope_apply(xr, rope_t);
            tq_rotate(xr, yr, sg, m, c.rot);
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
}

// ---------------------------------------------------------------------------
// Route (standalone call): grid = (ceil(G / 128), B * Hkv).  Each CTA stages
// its 128 groups' summary keys in shared memory, scores them against the
// aggregated rotated query, and the last CTA of a (b, h) selects.
// ---------------------------------------------------------------------------

template <int R>
__global__ void __launch_bounds__(kThreads) route_kernel(CacheView c, RouteArgs a, Tables tb) {
    extern __shared__ __align__(16) uint8_t s_dyn[];
    __shared__ __align__(16) float s_cb[hsq::kCodebookFloats];
    __shared__ __align__(16) float s_q[R][kDim];
    __shared__ SelectSmem s_ss;
    __shared__ int s_flag;

    const int bh = blockIdx.y, b = bh / c.Hkv, h = bh % c.Hkv;
    const int tid = threadIdx.x, hw = tid >> 4, l = hlane();
    uint32_t* s_keys = reinterpret_cast<uint32_t*>(s_dyn);
    uint8_t* s_codes = s_dyn + al16((size_t)c.G * 4);
    float* s_kn = reinterpret_cast<float*>(s_codes + kRouteGroupsPerCta * 48);
    uint8_t* s_cnt = reinterpret_cast<uint8_t*>(s_kn + kRouteGroupsPerCta);

    const int g_begin = blockIdx.x * kRouteGroupsPerCta;
    const int ng = min(c.G, g_begin + kRouteGroupsPerCta) - g_begin;
    // tier buffers: bh, except under per-query-head routing (run with R = 1)
    const size_t bb = R == 1 ? buf_head(c, b, h) : (size_t)bh;
    stage16(s_codes, c.l2_kc + (bb * c.G + g_begin) * 48, ng * 48);
    stage4(s_kn, c.l2_kn + bb * c.G + g_begin, ng);
    if (tid < hsq::kCodebookFloats / 4) cp_async16(s_cb + 4 * tid, tb.cb + 4 * tid);
    for (int i = tid; i < ng; i += kThreads) s_cnt[i] = __ldg(c.l2_cnt + (size_t)b * c.G + g_begin + i);
    float sg[8];
    load_signs_global(sg, c.signs);
    const int p = checked_pos(__ldcg(a.pos + b), tb, a.err);
    prepare_queries<R>(a.q + ((size_t)b * c.Hq + h * R) * kDim, p, sg, tb, s_q, nullptr, c.rot);
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
    const size_t base = (size_t)bh * c.G + g_begin;
    float qt[R][8];  // the rotated query heads (max aggregation)
#pragma unroll
    for (int j = 0; j < R; ++j) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            qt[j][k] = s_q[j][4 * l + k];
            qt[j][4 + k] = s_q[j][64 + 4 * l + k];
        }
    }
#pragma unroll 1
    for (int blk = 0; blk < ng; blk += 2 * kHalves) {
        const int ia = blk + hw, ib = ia + kHalves;
        const int ja = min(ia, ng - 1), jb = min(ib, ng - 1);
        float va[8], vb[8];
        unpack3_smem(s_codes + ja * 48, c3, 1.0f, va);
        unpack3_smem(s_codes + jb * 48, c3, 1.0f, vb);
        float sa, sb;
        if (a.agg_max) {  // per-head dots, then their maximum (a uniform branch)
            int idx;
            const float d = pair_dots<R>(qt, va, vb, idx);
            sa = idx < R ? d : -INFINITY;
            sb = (idx >= R) & (idx < 2 * R) ? d : -INFINITY;
#pragma unroll
            for (int o = 1; o < 16; o <<= 1) {
                sa = fmaxf(sa, __shfl_xor_sync(kFull, sa, o, 16));
                sb = fmaxf(sb, __shfl_xor_sync(kFull, sb, o, 16));
            }
        } else {
            route_pair(gq, va, vb, sa, sb);
        }
        if (l == 0) {
            if (ia < ng) a.scores[base + ia] = s_cnt[ja] > 0 ? s_kn[ja] * sa : -INFINITY;
            if (ib < ng) a.scores[base + ib] = s_cnt[jb] > 0 ? s_kn[jb] * sb : -INFINITY;
        }
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
    select_top_beta<kThreads>(s_keys, c.G, c.beta, a.sel + (size_t)bh * c.beta, s_ss);
    if (tid == 0) a.counters[bh] = 0;
}

// ---------------------------------------------------------------------------
// Fetch + dequantise (standalone): one CTA per (selected slot i, b*Hkv + h).
// ---------------------------------------------------------------------------

// Slot i of (b, h) holds group sel[b][h][i] (fetch), or g0 + i when sel is
// NULL (recover: keys stay pre-RoPE).  Outputs have nslot slots per (b, h).
struct FetchArgs {
    const int32_t* sel; float* k_out; float* v_out; uint8_t* valid; uint8_t* staging; int* err;
    int g0; int nslot;
};

template <int N>
__global__ void __launch_bounds__(kThreads) fetch_kernel(CacheView c, FetchArgs a, Tables tb) {
    __shared__ float s_cb[hsq::kCodebookFloats];
    __shared__ float s_sign[kDim];
    __shared__ __align__(16) uint8_t s_rec[N * 136];
    __shared__ int s_g;

    const int i = blockIdx.x, bh = blockIdx.y, b = bh / c.Hkv;
    const size_t bb = buf_head(c, b, bh % c.Hkv);  // tier buffers (bh unless routing per query head)
    const int hw = threadIdx.x >> 4, l = hlane();
    const unsigned m = half_mask();
    load_tables(s_cb, s_sign, tb, c.signs);
    if (threadIdx.x == 0) s_g = a.sel ? valid_sel(a.sel + (size_t)bh * c.beta, i, c.G, a.err) : a.g0 + i;
    __syncthreads();
    const int g = s_g;
    constexpr int kChunks = N * 136 / 16;
    uint4* srec = reinterpret_cast<uint4*>(s_rec);
    for (int k = threadIdx.x; k < kChunks; k += blockDim.x) {
        uint4 v = make_uint4(0, 0, 0, 0);
        if (g >= 0) v = __ldcg(reinterpret_cast<const uint4*>(c.l3 + (bb * c.G + g) * (N * 136)) + k);
        srec[k] = v;
        if (a.staging) reinterpret_cast<uint4*>(a.staging + ((size_t)bh * a.nslot + i) * (N * 136))[k] = v;
    }
    __syncthreads();
    if (hw >= N) return;
    float sg[8];
    load_signs(sg, s_sign);
    const int t = g * N + hw;
    const bool have = g >= 0 && t < c.T;
    const size_t oo = (((size_t)bh * a.nslot + i) * N + hw) * kDim;
    float kx[8], vx[8];
    if (have) {
        const float* c4 = s_cb;
        const float* norms = reinterpret_cast<const float*>(s_rec + N * 128);
        const uint16_t* kr = reinterpret_cast<const uint16_t*>(s_rec + hw * 64);
        const uint16_t* vr = reinterpret_cast<const uint16_t*>(s_rec + N * 64 + hw * 64);
        unpack4(kr[l], kr[16 + l], c4, 1.0f, kx);
        unpack4(vr[l], vr[16 + l], c4, 1.0f, vx);
        if (c.rot) {
            fwht(kx, m);
            fwht(vx, m);
        }
        const float sc = c.rot ? kRsqrtD : 1.f;
        const float kn = norms[hw] * sc, vn = norms[N + hw] * sc;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            kx[q] *= sg[q] * kn;
            vx[q] *= sg[q] * vn;
        }
        if (a.sel) rope(kx, t, tb);
    } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) kx[q] = vx[q] = 0.f;
    }
    if (a.k_out) store_f32x8(a.k_out + oo, kx);
    if (a.v_out) store_f32x8(a.v_out + oo, vx);
    if (a.valid && l == 0)
        a.valid[((size_t)bh * a.nslot + i) * N + hw] = (uint8_t)(have && !in_l1(c, b, t));
}

}  // namespace

// ===========================================================================
// Host side: shared helpers and entry points (struct hsq_ctx: hsq_ctx.h).
// ===========================================================================

namespace hsq {

hsq_status fail(hsq_ctx* ctx, hsq_status st, const std::string& msg) {
    if (ctx) ctx->last_error = msg;
    set_process_error(msg);
    return st;
}

hsq_status cuda_fail(hsq_ctx* ctx, cudaError_t e, const char* where) {
    return fail(ctx, HSQ_ERR_CUDA, std::string(where) + ": " + cudaGetErrorString(e));
}

namespace {
std::mutex g_smem_mu;
std::vector<std::pair<std::pair<const void*, int>, size_t>> g_smem_limits;
std::vector<std::pair<const void*, int>> g_big_clusters;
}  // namespace

// The dynamic shared-memory ceiling is a property of the kernel (per device),
// shared by every context of the process: only ever raise it.
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

cudaError_t allow_big_clusters(const void* fn, int device) {
    std::lock_guard<std::mutex> lk(g_smem_mu);
    for (auto& e : g_big_clusters)
        if (e.first == fn && e.second == device) return cudaSuccess;
    cudaError_t err = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (err == cudaSuccess) g_big_clusters.push_back({fn, device});
    return err;
}

}  // namespace hsq

namespace {

using hsq::cuda_fail;
using hsq::fail;
using hsq::raise_smem_limit;

#define HSQ_CUDA(ctx, call)                                   \
    do {                                                      \
        cudaError_t e_ = (call);                              \
        if (e_ != cudaSuccess) return cuda_fail(ctx, e_, #call); \
    } while (0)

bool r_supported(int r) { return r == 1 || r == 2 || r == 4 || r == 5 || r == 8; }

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
    switch (v.Hq / v.Hkv) {  // 1 under per-query-head routing
        case 1: return launch_route<1>(ctx, v, a, st);
        case 2: return launch_route<2>(ctx, v, a, st);
        case 4: return launch_route<4>(ctx, v, a, st);
        case 5: return launch_route<5>(ctx, v, a, st);
        case 8: return launch_route<8>(ctx, v, a, st);
    }
    return HSQ_ERR_UNSUPPORTED;
}

hsq_status decode_run(hsq_ctx* ctx, const hsq_cache* cache, const float* q, const int32_t* pos, int32_t* sel,
                      float* out, bool route, bool from_staging, cudaStream_t st, bool* launched) {
    switch (ctx->cfg.route_per_head ? 1 : ctx->r) {  // per query head: one head per view head
        case 1: return hsq::decode_run_r1(ctx, cache, q, pos, sel, out, route, from_staging, st, launched);
        case 2: return hsq::decode_run_r2(ctx, cache, q, pos, sel, out, route, from_staging, st, launched);
        case 4: return hsq::decode_run_r4(ctx, cache, q, pos, sel, out, route, from_staging, st, launched);
        case 5: return hsq::decode_run_r5(ctx, cache, q, pos, sel, out, route, from_staging, st, launched);
        case 8: return hsq::decode_run_r8(ctx, cache, q, pos, sel, out, route, from_staging, st, launched);
    }
    return fail(ctx, HSQ_ERR_UNSUPPORTED, "unsupported head ratio");
}

// q, pos, sel and out may be device memory or page-locked host memory mapped
// into the device address space; anything else (pageable host memory) is
// refused here rather than faulting in a kernel.
hsq_status check_accessible(hsq_ctx* ctx, const void* p, const char* what) {
    for (const void* q : ctx->accessible)
        if (q == p) return HSQ_OK;
    cudaPointerAttributes pa;
    cudaError_t e = cudaPointerGetAttributes(&pa, p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(ctx, HSQ_ERR_INVALID, std::string(what) + " is not a device or page-locked host pointer");
    }
    const bool ok = pa.type == cudaMemoryTypeDevice || pa.type == cudaMemoryTypeManaged ||
                    (pa.type == cudaMemoryTypeHost && pa.devicePointer == p);
    if (!ok) return fail(ctx, HSQ_ERR_INVALID, std::string(what) + " is not device-accessible at this address");
    if (ctx->accessible.size() >= 64) ctx->accessible.erase(ctx->accessible.begin());
    ctx->accessible.push_back(p);
    return HSQ_OK;
}

hsq_status check_io(hsq_ctx* ctx, const float* q, const int32_t* pos, const int32_t* sel, const float* out) {
    hsq_status st;
    if ((st = check_accessible(ctx, q, "q")) != HSQ_OK) return st;
    if ((st = check_accessible(ctx, pos, "pos")) != HSQ_OK) return st;
    if (sel && (st = check_accessible(ctx, sel, "sel")) != HSQ_OK) return st;
    if (out && (st = check_accessible(ctx, out, "out")) != HSQ_OK) return st;
    return HSQ_OK;
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

// Encode of a layer (hsq_encode); with pf, also the prefill's K/V operand images.
hsq_status encode_run(hsq_ctx* ctx, const hsq_cache* cache, const void* K, const void* V, hsq_dtype dtype,
                      cudaStream_t s, const hsq::PrefillImages* pf) {
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
    CacheView v = make_view(ctx, cache);
    if (pf && (size_t)v.G * v.N < (size_t)pf->nkt * 64) {
        // key rows past the encode's groups: the attention reads them as zeros
        HSQ_CUDA(ctx, cudaMemsetAsync(pf->kh, 0, pf->bytes - (size_t)(pf->kh - pf->qh), s));
    }
    if (v.hot_tag)  // the hot-group table holds copies of the old records: empty it
        HSQ_CUDA(ctx, cudaMemsetAsync(v.hot_tag, 0xFF, (size_t)v.B * v.Hkv * (v.hot_mask + 1) * 4, s));
    l1_index_kernel<<<v.B, 1024, 0, s>>>(v, cache->l1_pos, cache->l1_count, ctx->d_prefix, ctx->d_err);
    const bool grow = ctx->cfg.l1_recent > 0 && cache->win_kv && cache->gsum;
    EncodeOut o{cache->l1_kc, cache->l1_vc, cache->l1_kn, cache->l1_vn, cache->l2_kc, cache->l2_vc,
                cache->l2_kn, cache->l2_vn, cache->l2_cnt, cache->l3, ctx->d_prefix,
                grow ? cache->win_kv : nullptr, grow ? cache->gsum : nullptr, ctx->cfg.l1_recent,
                pf ? pf->kh : nullptr, pf ? pf->kl : nullptr, pf ? pf->vt : nullptr, pf ? pf->nkt : 0,
                ctx->cfg.qjl ? ctx->d_qjl_kc : nullptr};
    const Tables tb = make_tables(ctx);
    using EncodeFn = void (*)(CacheView, EncodeOut, const void*, const void*, Tables);
    const bool bf = dtype == HSQ_DTYPE_BF16;
    EncodeFn fn;  // the variant of the block size, input type and codec
    if (pf) {     // prefill: bf16 inputs
        if (v.N == 16) fn = v.rot ? encode_kernel<16, true, true, true> : encode_kernel<16, true, false, true>;
        else fn = v.rot ? encode_kernel<8, true, true, true> : encode_kernel<8, true, false, true>;
    } else if (v.N == 16) {
        fn = v.rot ? (bf ? encode_kernel<16, true, true> : encode_kernel<16, false, true>)
                   : (bf ? encode_kernel<16, true, false> : encode_kernel<16, false, false>);
    } else {
        fn = v.rot ? (bf ? encode_kernel<8, true, true> : encode_kernel<8, false, true>)
                   : (bf ? encode_kernel<8, true, false> : encode_kernel<8, false, false>);
    }
    const size_t dyn = enc_dyn_smem(v.N);
    HSQ_CUDA(ctx, raise_smem_limit((const void*)fn, ctx->device, dyn));
    fn<<<dim3((v.G + kEncGroups - 1) / kEncGroups, v.Hkv, v.B), v.N * 32, dyn, s>>>(v, o, K, V, tb);
    if (ctx->cfg.qjl) {  // TQ-QKV: the key-residual sketches (after the L1 slot prefix is known)
        uint4* sf = reinterpret_cast<uint4*>(ctx->d_qjl_sb);
        qjl_pack_kernel<<<16, 256, 0, s>>>(cache->qjl_s, cache->signs, v.rot, sf);
        const SketchOut so{sf, cache->l1_qs, cache->l1_qn, cache->l3_qs, cache->l3_qn, ctx->d_qjl_kc};
        const dim3 g3((v.T + kQjlTok - 1) / kQjlTok, v.Hkv, v.B), g1((v.max_l1 + 15) / 16, v.Hkv, v.B);
        if (v.N == 16) {
            if (bf) qjl_kernel<16, true><<<g3, kQjlThreads, 0, s>>>(v, so, K, tb);
            else qjl_kernel<16, false><<<g3, kQjlThreads, 0, s>>>(v, so, K, tb);
        } else {
            if (bf) qjl_kernel<8, true><<<g3, kQjlThreads, 0, s>>>(v, so, K, tb);
            else qjl_kernel<8, false><<<g3, kQjlThreads, 0, s>>>(v, so, K, tb);
        }
        if (bf) qjl_l1_kernel<true><<<g1, kQjlThreads, 0, s>>>(v, so, K, tb);
        else qjl_l1_kernel<false><<<g1, kQjlThreads, 0, s>>>(v, so, K, tb);
    }
    return after_launch(ctx, "encode");
}

void free_ctx(hsq_ctx* c) {
    cudaFree(c->d_cb); cudaFree(c->d_rope_hi); cudaFree(c->d_rope_lo); cudaFree(c->d_scores);
    cudaFree(c->d_route_ctr); cudaFree(c->d_prefix); cudaFree(c->d_err); cudaFree(c->d_qjl_sb);
    cudaFree(c->d_qjl_kc);
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
    // one routing row per KV head, or per query head under per-query-head routing
    const size_t bh = (size_t)cfg->max_batch * (cfg->route_per_head ? cfg->n_q_heads : cfg->n_kv_heads);

    if ((e = cudaMalloc(&c->d_cb, sizeof(cb))) != cudaSuccess) return bail(e, "cudaMalloc(codebook)");
    if ((e = cudaMalloc(&c->d_rope_hi, hi.size() * 4)) != cudaSuccess) return bail(e, "cudaMalloc(rope)");
    if ((e = cudaMalloc(&c->d_rope_lo, lo.size() * 4)) != cudaSuccess) return bail(e, "cudaMalloc(rope)");
    if ((e = cudaMalloc(&c->d_scores, bh * c->G_max * 4)) != cudaSuccess) return bail(e, "cudaMalloc(scores)");
    if ((e = cudaMalloc(&c->d_route_ctr, bh * 4)) != cudaSuccess) return bail(e, "cudaMalloc(counters)");
    if ((e = cudaMalloc(&c->d_prefix, (size_t)cfg->max_batch * c->W_max * 4)) != cudaSuccess)
        return bail(e, "cudaMalloc(prefix)");
    if ((e = cudaMalloc(&c->d_err, 4)) != cudaSuccess) return bail(e, "cudaMalloc(err)");
    if (cfg->qjl && (e = cudaMalloc(&c->d_qjl_sb, hsq::kDim * hsq::kDim * 4)) != cudaSuccess)
        return bail(e, "cudaMalloc(sketch matrix)");
    if (cfg->qjl && (e = cudaMalloc(&c->d_qjl_kc, (size_t)cfg->max_batch * cfg->n_kv_heads * c->G_max *
                                                      cfg->group_n * 68)) != cudaSuccess)
        return bail(e, "cudaMalloc(key codes)");
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
    return encode_run(ctx, cache, K, V, dtype, reinterpret_cast<cudaStream_t>(stream), nullptr);
}

hsq_status hsq_prefill_workspace_size(const hsq_ctx* ctx, int B, int T, size_t* bytes) {
    if (!ctx || !bytes) return fail(nullptr, HSQ_ERR_INVALID, "ctx or bytes is NULL");
    if (B < 1 || T < 1) return fail(nullptr, HSQ_ERR_INVALID, "B and T must be positive");
    *bytes = hsq::prefill_images(nullptr, B, ctx->cfg.n_q_heads, ctx->cfg.n_kv_heads, T).bytes;
    return HSQ_OK;
}

hsq_status hsq_prefill(hsq_ctx* ctx, const hsq_cache* cache, const void* Q, const void* K, const void* V, int B,
                       int T, float* out, void* workspace, size_t workspace_bytes, hsq_stream_t stream) {
    if (!ctx) return fail(nullptr, HSQ_ERR_INVALID, "context is NULL");
    if (!Q || !K || !V || !out || !workspace) return fail(ctx, HSQ_ERR_INVALID, "Q, K, V, out or workspace is NULL");
    if (B < 1 || T < 1 || B > ctx->cfg.max_batch || T > ctx->cfg.max_pos)
        return fail(ctx, HSQ_ERR_INVALID, "B or T outside the context's limits (max_batch, max_pos)");
    if (cache && (cache->B != B || cache->T != T)) return fail(ctx, HSQ_ERR_INVALID, "cache B / T differ from B / T");
    if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
        return fail(ctx, HSQ_ERR_INVALID, "workspace must be 256-byte aligned");
    const hsq::PrefillImages im = hsq::prefill_images(workspace, B, ctx->cfg.n_q_heads, ctx->cfg.n_kv_heads, T);
    if (workspace_bytes < im.bytes) return fail(ctx, HSQ_ERR_INVALID, "workspace smaller than hsq_prefill_workspace_size");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    hsq_status st;
    if (cache) {
        st = encode_run(ctx, cache, K, V, HSQ_DTYPE_BF16, s, &im);  // the encode writes the K/V operands
    } else {
        st = hsq::prefill_prep_kv(ctx, im, K, V, B, T, s);
    }
    if (st != HSQ_OK) return st;
    if ((st = hsq::prefill_prep_q(ctx, im, Q, B, T, s)) != HSQ_OK) return st;
    return hsq::prefill_attention(ctx, im, out, B, T, s);
}

hsq_status hsq_append(hsq_ctx* ctx, hsq_cache* cache, const void* k, const void* v, hsq_dtype dtype,
                      hsq_stream_t stream) {
    hsq_status st = check_common(ctx, cache);
    if (st != HSQ_OK) return st;
    if (!k || !v) return fail(ctx, HSQ_ERR_INVALID, "k or v is NULL");
    if (dtype != HSQ_DTYPE_F32 && dtype != HSQ_DTYPE_BF16) return fail(ctx, HSQ_ERR_INVALID, "bad dtype");
    if (ctx->cfg.qjl) return fail(ctx, HSQ_ERR_UNSUPPORTED, "hsq_append does not sketch key residuals (cfg.qjl)");
    const int recent = ctx->cfg.l1_recent;
    if (recent < 1) return fail(ctx, HSQ_ERR_INVALID, "the context has no recent window (l1_recent = 0)");
    if (!cache->win_kv || !cache->gsum) return fail(ctx, HSQ_ERR_INVALID, "win_kv or gsum is NULL");
    const int cap = cache->t_cap > 0 ? cache->t_cap : cache->T;
    if (cache->T >= cap) return fail(ctx, HSQ_ERR_INVALID, "the cache is full (T == t_cap)");
    if (cache->T >= ctx->cfg.max_pos) return fail(ctx, HSQ_ERR_INVALID, "position T reaches max_pos");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const CacheView vw = make_view(ctx, cache);
    if (vw.Hkv > 32) return fail(ctx, HSQ_ERR_UNSUPPORTED, "hsq_append handles at most 32 KV heads");
    EncodeOut o{cache->l1_kc, cache->l1_vc, cache->l1_kn, cache->l1_vn, cache->l2_kc, cache->l2_vc,
                cache->l2_kn, cache->l2_vn, cache->l2_cnt, cache->l3, nullptr, cache->win_kv, cache->gsum,
                recent};
    const Tables tb = make_tables(ctx);
    const bool bf = dtype == HSQ_DTYPE_BF16;
    const int threads = 32 * std::min(vw.Hkv + 1, 32), sinks = ctx->cfg.l1_sinks;  // + the bookkeeping warp
    int32_t* pos = cache->l1_pos;
    int32_t* cnt = cache->l1_count;
    uint32_t* bm = cache->l1_bitmap;
    if (vw.N == 16) {
        if (bf) append_kernel<16, true><<<vw.B, threads, 0, s>>>(vw, o, pos, cnt, bm, k, v, tb, sinks, recent, ctx->d_err);
        else append_kernel<16, false><<<vw.B, threads, 0, s>>>(vw, o, pos, cnt, bm, k, v, tb, sinks, recent, ctx->d_err);
    } else {
        if (bf) append_kernel<8, true><<<vw.B, threads, 0, s>>>(vw, o, pos, cnt, bm, k, v, tb, sinks, recent, ctx->d_err);
        else append_kernel<8, false><<<vw.B, threads, 0, s>>>(vw, o, pos, cnt, bm, k, v, tb, sinks, recent, ctx->d_err);
    }
    st = after_launch(ctx, "append");
    if (st == HSQ_OK) cache->T += 1;
    return st;
}

hsq_status hsq_route(hsq_ctx* ctx, const hsq_cache* cache, const float* q, const int32_t* pos,
                     int32_t* sel, float* scores_opt, hsq_stream_t stream) {
    hsq_status st = check_common(ctx, cache);
    if (st != HSQ_OK) return st;
    if (!q || !pos || !sel) return fail(ctx, HSQ_ERR_INVALID, "q, pos or sel is NULL");
    if ((st = check_io(ctx, q, pos, sel, nullptr)) != HSQ_OK) return st;
    CacheView v = make_sel_view(ctx, cache);
    RouteArgs a{q, pos, sel, scores_opt ? scores_opt : ctx->d_scores, ctx->d_route_ctr, ctx->d_err,
                ctx->cfg.route_max};
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
    CacheView v = make_sel_view(ctx, cache);
    FetchArgs a{sel, k_out_opt, v_out_opt, valid_opt, cache->staging, ctx->d_err, 0, v.beta};
    dim3 grid(v.beta, v.B * v.Hkv);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (v.N == 16) fetch_kernel<16><<<grid, kThreads, 0, s>>>(v, a, make_tables(ctx));
    else fetch_kernel<8><<<grid, kThreads, 0, s>>>(v, a, make_tables(ctx));
    return after_launch(ctx, "fetch_dequant");
}

hsq_status hsq_recover(hsq_ctx* ctx, const hsq_cache* cache, int g0, int ng, float* k_out_opt,
                       float* v_out_opt, hsq_stream_t stream) {
    hsq_status st = check_common(ctx, cache);
    if (st != HSQ_OK) return st;
    const int groups = hsq::groups_of(cache->T, ctx->cfg.group_n);
    if (g0 < 0 || ng < 1 || (long long)g0 + ng > groups)
        return fail(ctx, HSQ_ERR_INVALID, "groups [g0, g0 + ng) must lie in [0, ceil(T / N))");
    if (!k_out_opt && !v_out_opt) return fail(ctx, HSQ_ERR_INVALID, "no output");
    if (k_out_opt && (st = check_accessible(ctx, k_out_opt, "k_out")) != HSQ_OK) return st;
    if (v_out_opt && (st = check_accessible(ctx, v_out_opt, "v_out")) != HSQ_OK) return st;
    CacheView v = make_view(ctx, cache);
    FetchArgs a{nullptr, k_out_opt, v_out_opt, nullptr, nullptr, ctx->d_err, g0, ng};
    dim3 grid(ng, v.B * v.Hkv);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (v.N == 16) fetch_kernel<16><<<grid, kThreads, 0, s>>>(v, a, make_tables(ctx));
    else fetch_kernel<8><<<grid, kThreads, 0, s>>>(v, a, make_tables(ctx));
    return after_launch(ctx, "recover");
}

hsq_status hsq_decode_attn(hsq_ctx* ctx, const hsq_cache* cache, const float* q, const int32_t* pos,
                           const int32_t* sel, float* out, int flags, hsq_stream_t stream) {
    hsq_status st = check_common(ctx, cache);
    if (st != HSQ_OK) return st;
    if (!q || !pos || !sel || !out) return fail(ctx, HSQ_ERR_INVALID, "q, pos, sel or out is NULL");
    if ((st = check_io(ctx, q, pos, sel, out)) != HSQ_OK) return st;
    if (flags & ~HSQ_ATTN_FROM_STAGING) return fail(ctx, HSQ_ERR_INVALID, "unknown flags");
    const bool staged = (flags & HSQ_ATTN_FROM_STAGING) != 0;
    if (staged && !cache->staging) return fail(ctx, HSQ_ERR_INVALID, "staging is NULL");
    if (hsq::fault_mask() & HSQ_FAULT_FETCH) return fail(ctx, HSQ_ERR_CUDA, "injected fetch failure");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    bool launched = false;
    hsq_status st2 = decode_run(ctx, cache, q, pos, const_cast<int32_t*>(sel), out, false, staged, s, &launched);
    if (st2 == HSQ_OK && !launched)
        return fail(ctx, HSQ_ERR_UNSUPPORTED, "decode kernel cannot be launched for this cache shape");
    return st2;
}

hsq_status hsq_decode_step(hsq_ctx* ctx, const hsq_cache* cache, const float* q, const int32_t* pos,
                           int32_t* sel, float* out, hsq_stream_t stream) {
    hsq_status st = check_common(ctx, cache);
    if (st != HSQ_OK) return st;
    if (!q || !pos || !sel || !out) return fail(ctx, HSQ_ERR_INVALID, "q, pos, sel or out is NULL");
    if ((st = check_io(ctx, q, pos, sel, out)) != HSQ_OK) return st;
    if (hsq::fault_mask() & HSQ_FAULT_FETCH) return fail(ctx, HSQ_ERR_CUDA, "injected fetch failure");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    bool fused = false;
    if (!ctx->cfg.route_max) {  // (the fused kernel routes by the sum over the query heads)
        st = decode_run(ctx, cache, q, pos, sel, out, true, false, s, &fused);
        if (st != HSQ_OK || fused) return st;
    }
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
// exits), the codebook travels by value in the kernel's parameters, and the
// query's RoPE angles are evaluated in float64 inside the kernel instead of
// being read from a context's tables.
// ===========================================================================

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[HSQ_NOALLOC_SCRATCH_BYTES];

struct NoallocCodebook { float v[hsq::kCodebookFloats]; };

constexpr int kNoallocMaxDevices = 64;
std::mutex g_noalloc_mu;
// per device: the scratch array's device address and the CUDA context it was
// looked up in (a device reset makes a new context and reloads the module)
unsigned char* g_noalloc_ptr[kNoallocMaxDevices] = {};
unsigned long long g_noalloc_ctx[kNoallocMaxDevices] = {};
bool g_noalloc_have_cb = false;
NoallocCodebook g_noalloc_cb;

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
__global__ void __launch_bounds__(kThreads) route_noalloc_kernel(CacheView c, RouteArgs a, double theta,
                                                                  int max_pos, NoallocCodebook cb) {
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
    for (int i = threadIdx.x; i < hsq::kCodebookFloats; i += blockDim.x) s_cb[i] = cb.v[i];
    for (int i = threadIdx.x; i < kDim; i += blockDim.x) s_sign[i] = c.signs ? (float)c.signs[i] : 1.f;
    __syncthreads();
    float sg[8];
    load_signs(sg, s_sign);

    if (hw < R) {
        const int j = h * R + hw;
        float x[8];
        load_f32x8(a.q + ((size_t)b * c.Hq + j) * kDim, x);
        // out-of-range positions are clamped to [0, max_pos) as hsq_route clamps
        // them (this entry point has no device error word to report them in)
        rope_f64(x, min(max(__ldg(a.pos + b), 0), max_pos - 1), theta);
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] *= sg[i];
        if (c.rot) fwht(x, m);
        const float sc = c.rot ? kRsqrtD : 1.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            s_q[hw][4 * l + k] = x[k] * sc;
            s_q[hw][64 + 4 * l + k] = x[4 + k] * sc;
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

// The unique id of the calling thread's current CUDA context (0 when none is
// current or the driver does not say), through driver entry points looked up
// once, so the library needs no link to the driver library.
unsigned long long current_context_id() {
    using GetCurrent = CUresult (*)(CUcontext*);
    using GetId = CUresult (*)(CUcontext, unsigned long long*);
    static GetCurrent get_current = nullptr;
    static GetId get_id = nullptr;
    static bool looked_up = false;
    if (!looked_up) {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &qr) == cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<GetCurrent>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &qr) == cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<GetId>(f);
        looked_up = true;
    }
    CUcontext cx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&cx) != CUDA_SUCCESS || !cx || get_id(cx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// Set-up of the current device: the scratch array's device address (a
// host-side use of the symbol name itself would not be a device address).
// Done on the first call on a device, and again when the device's CUDA
// context has changed since (after a device reset the module is reloaded
// and the array has a new address).  Synchronous on first use of a context,
// so such a call must not run under stream capture.  The codebook is
// computed once per process on the host and passed by value.
hsq_status noalloc_setup(unsigned char** scratch, NoallocCodebook* cb) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(nullptr, e, "cudaGetDevice");
    if (dev < 0 || dev >= kNoallocMaxDevices) return fail(nullptr, HSQ_ERR_UNSUPPORTED, "device ordinal above 63");
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_have_cb) {
        hsq::device_codebook(g_noalloc_cb.v);
        g_noalloc_have_cb = true;
    }
    const unsigned long long ctx_id = current_context_id();
    if (!g_noalloc_ptr[dev] || ctx_id == 0 || ctx_id != g_noalloc_ctx[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_fail(nullptr, e, "cudaGetSymbolAddress(scratch)");
        g_noalloc_ptr[dev] = static_cast<unsigned char*>(p);
        g_noalloc_ctx[dev] = current_context_id();  // the context the lookup ran in
    }
    *scratch = g_noalloc_ptr[dev];
    *cb = g_noalloc_cb;
    return HSQ_OK;
}

template <int R>
hsq_status launch_route_noalloc(const CacheView& v, const RouteArgs& a, double theta, int max_pos,
                                const NoallocCodebook& cb, cudaStream_t st, int dev) {
    const size_t smem = (size_t)v.G * 4;
    if (smem > 48 * 1024) {
        cudaError_t e = raise_smem_limit((const void*)route_noalloc_kernel<R>, dev, smem);
        if (e != cudaSuccess) return cuda_fail(nullptr, e, "cudaFuncSetAttribute");
    }
    dim3 grid((v.G + kRouteGroupsPerCta - 1) / kRouteGroupsPerCta, v.B * v.Hkv);
    route_noalloc_kernel<R><<<grid, kThreads, smem, st>>>(v, a, theta, max_pos, cb);
    return HSQ_OK;
}

}  // namespace

extern "C" hsq_status hsq_route_noalloc(const hsq_config* cfg, const hsq_cache* cache, const float* q,
                                        const int32_t* pos, int32_t* sel, hsq_stream_t stream) {
    std::string why = hsq::check_config(cfg);
    if (!why.empty()) return fail(nullptr, HSQ_ERR_INVALID, why);
    why = hsq::check_cache_shape(cfg, cache);
    if (!why.empty()) return fail(nullptr, HSQ_ERR_INVALID, why);
    if (cfg->route_max || cfg->route_per_head)
        return fail(nullptr, HSQ_ERR_UNSUPPORTED, "hsq_route_noalloc routes by the sum over the query heads only");
    if (!q || !pos || !sel) return fail(nullptr, HSQ_ERR_INVALID, "q, pos or sel is NULL");
    const int r = cfg->n_q_heads / cfg->n_kv_heads;
    if (!r_supported(r)) return fail(nullptr, HSQ_ERR_UNSUPPORTED, "r = Hq/Hkv must be 1, 2, 4, 5 or 8");
    const size_t bh = (size_t)cache->B * cfg->n_kv_heads;
    const int cap = cache->t_cap > 0 ? cache->t_cap : cache->T;  // the layout's capacity
    const size_t G = (size_t)hsq::groups_of(cap, cfg->group_n);
    const size_t ticket_bytes = (bh * 4 + 255) / 256 * 256;
    if (ticket_bytes + bh * G * 4 > (size_t)HSQ_NOALLOC_SCRATCH_BYTES)
        return fail(nullptr, HSQ_ERR_INVALID,
                    "B * n_kv_heads * ceil(T / group_n) too large for the fixed 4 MiB scratch of hsq_route_noalloc");
    if (G * 4 > 200 * 1024) return fail(nullptr, HSQ_ERR_INVALID, "ceil(T / group_n) above 51200");
    unsigned char* scratch = nullptr;
    NoallocCodebook cb;
    hsq_status st = noalloc_setup(&scratch, &cb);
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
    v.max_l1 = cfg->max_l1; v.W = hsq::bitmap_words(cap); v.cap = cap;
    v.l2_kc = cache->l2_kc; v.l2_kn = cache->l2_kn; v.l2_cnt = cache->l2_cnt;
    v.rot = cfg->codec == HSQ_CODEC_PLAIN ? 0 : 1;
    v.signs = v.rot ? cache->signs : nullptr;
    RouteArgs a{q, pos, sel, reinterpret_cast<float*>(scratch + ticket_bytes),
                reinterpret_cast<int*>(scratch), nullptr};
    switch (r) {
        case 1: st = launch_route_noalloc<1>(v, a, cfg->rope_theta, cfg->max_pos, cb, s, dev); break;
        case 2: st = launch_route_noalloc<2>(v, a, cfg->rope_theta, cfg->max_pos, cb, s, dev); break;
        case 4: st = launch_route_noalloc<4>(v, a, cfg->rope_theta, cfg->max_pos, cb, s, dev); break;
        case 5: st = launch_route_noalloc<5>(v, a, cfg->rope_theta, cfg->max_pos, cb, s, dev); break;
        default: st = launch_route_noalloc<8>(v, a, cfg->rope_theta, cfg->max_pos, cb, s, dev); break;
    }
    if (st != HSQ_OK) return st;
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(nullptr, e, "route_noalloc");
    return HSQ_OK;
}
