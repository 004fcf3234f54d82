// Prefill: the prompt's dense causal attention on the tensor cores.
//
// "Tamarin (HSQ)" technical summary, section 4 (results): compressing the
// prompt's K/V costs a prefill overhead of 1.2-1.3x at 32K.  The prompt's
// attention itself is the model's ordinary causal softmax attention over
// RoPE'd queries and keys (GQA, scale 1/sqrt(d)); HSQ only decides what is
// kept for decoding.  hsq_prefill runs the encode of K/V (hsq_encode's
// kernel, which then also writes the attention's K/V operands, so K/V are
// read once) and this attention.
//
// Operands.  Queries and keys are RoPE'd in fp32 and each split into two
// bf16 terms x = hi + lo; logits use hi.hi + lo.hi + hi.lo (three MMAs, the
// dropped lo.lo term is below 2^-16 of the product), probabilities p =
// ph + pl multiply the bf16 values (exact: the inputs are bf16).  So the
// tensor cores give fp32-level logits and outputs.  Every operand tile is
// stored in global memory as the exact shared-memory image the MMA reads
// (K-major, 128-byte swizzle), so one 1-D bulk copy per tile fills shared
// memory:
//   Q  [B][Hq][ceil(T/128)] images of 128 rows x 128 dims (hi and lo, 32 KB each)
//   K  [B][Hkv][2 ceil(T/128)] images of 64 rows x 128 dims (hi and lo, 16 KB each)
//   Vt [B][Hkv][2 ceil(T/128)] images of 128 dims x 64 keys (16 KB), V transposed
//      so that it is the K-major B operand of P V.
// Rows past T are zero.
//
// Attention kernel: one CTA per (128-query tile, query head, sequence), warp
// specialised.  The query tile is loaded once and moved by the softmax warps
// into TMEM columns 384-511 (hi, lo; row = lane, dims in pairs along the
// columns), so the S products take their A operand from tensor memory and
// only the key tiles are read from shared memory.  Two producer warps, one
// thread each: warp 8 loads the key tiles and issues S = Q K^T of tile k
// (128 x 64, into TMEM columns 0-63 or 64-127 in turn) as soon as the tile's
// keys have landed and the softmax has read the buffer's previous S; warp 9
// loads the value tiles and, once the
// softmax has written P of tile k, issues O_half += P_half V_half for both
// key halves (TMEM columns 128-255 and 256-383).  Each refills its stage when
// the MMA that read it completed.  Warps 0-7 run the softmax: query row r of
// the tile is TMEM lane r (a warp reaches only its quarter of the lanes,
// 32 (w & 3) .. + 31) and warp w handles the key half w >> 2 of every 64-key
// tile, so two threads share a row; each key half keeps its own online
// softmax (log2 domain: the queries carry the scale log2(e) / sqrt(d); its
// running maximum is raised only when a logit exceeds it by more than 8,
// then its O in TMEM is rescaled) and its own accumulator, combined once at
// the end; only the two diagonal tiles apply the causal mask.  The roles
// meet only on mbarriers (S full / S read / P full / O done, two of each,
// one per buffer), so the S of the next tiles runs on the tensor cores while
// the softmax of this one runs, and P is double-buffered.  The output is the
// combined O / l in fp32.
#include <cuda_runtime.h>

#include <cstdint>

#include "hsq_ctx.h"
#include "hsq_device.cuh"
#include "hsq_tc.cuh"

namespace {

using namespace hsq_tc;

constexpr int kPfRows = 128;                          // query rows per CTA (TMEM lanes)
constexpr int kPfKeys = 64;                           // keys per tile
constexpr int kPfSoftThreads = 256;                   // softmax warps 0-7
constexpr int kPfThreads = kPfSoftThreads + 64;       // + the two producer warps
constexpr uint32_t kQImg = kPfRows * kDim * 2;        // 32 KB
constexpr uint32_t kKImg = kPfKeys * kDim * 2;        // 16 KB
constexpr uint32_t kVImg = kDim * kPfKeys * 2;        // 16 KB
constexpr uint32_t kPImg = kPfRows * kPfKeys * 2;     // 16 KB
constexpr uint32_t kOffQh = 0, kOffQl = kQImg, kOffK = 2 * kQImg;   // K stage b: Kh | Kl
constexpr uint32_t kOffV = kOffK + 2 * 2 * kKImg;                    // V stage b
constexpr uint32_t kOffP = kOffV + 2 * kVImg;                        // P buffer b: Ph | Pl
constexpr uint32_t kOffBar = kOffP + 2 * 2 * kPImg;
// barriers (8 bytes each): q | k[2] | v[2] | s_full[2] | s_free[2] | p_full[2] | o_done[2]; TMEM address
constexpr int kNumBars = 14;
constexpr uint32_t kPfSmem = kOffBar + 8 * kNumBars + 8 + 1024;
constexpr uint32_t kTmemCols = 512;  // S buffers: 0-63, 64-127; O of key half k: 128 + 128 k; Q hi 384, lo 448
constexpr uint32_t kTmQh = 384, kTmQl = 448;

struct PrefillArgs {
    const uint8_t* qh; const uint8_t* ql; const uint8_t* kh; const uint8_t* kl; const uint8_t* vt;
    float* out;  // [B][Hq][T][128]
    int* err;
    int Hq, Hkv, T, nqt, nkt;
};

__global__ void __launch_bounds__(kPfThreads, 1) prefill_attn_kernel(PrefillArgs a) {
    extern __shared__ uint8_t pf_raw[];
    const uint32_t raw = smem_addr(pf_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = pf_raw + (base - raw);
    const int tid = threadIdx.x, warp = tid >> 5, lanei = tid & 31;
    const int qt = a.nqt - 1 - (int)blockIdx.x;    // the longest rows first
    const int j = blockIdx.y, b = blockIdx.z;
    const int h = j / (a.Hq / a.Hkv);
    const uint32_t bar0 = base + kOffBar;
    const uint32_t bar_q = bar0, bar_k = bar0 + 8, bar_v = bar0 + 24, s_full = bar0 + 40, s_free = bar0 + 56;
    const uint32_t p_full = bar0 + 72, o_done = bar0 + 88, q_tm = bar0 + 104, slot = bar0 + 8 * kNumBars;
    const int nkv = 2 * qt + 2;  // key tiles up to the diagonal

    if (tid == 0) {
        mbar_init(bar_q, 1);
        mbar_init(q_tm, kPfSoftThreads);
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar_k + 8 * i, 1);
            mbar_init(bar_v + 8 * i, 1);
            mbar_init(s_full + 8 * i, 1);
            mbar_init(s_free + 8 * i, kPfSoftThreads);
            mbar_init(p_full + 8 * i, kPfSoftThreads);
            mbar_init(o_done + 8 * i, 1);
        }
        mbar_init_fence();
    }
    if (warp == 0) {
        tmem_alloc(slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(gbase + kOffBar + 8 * kNumBars);
    bool ok = true;

    if (warp >= kPfSoftThreads / 32) {
        // ---- producers, one thread each: warp 8 the keys and S, warp 9 the values and P V ----
        const size_t kv0 = ((size_t)b * a.Hkv + h) * a.nkt;
        if (warp == kPfSoftThreads / 32 && lanei == 0) {
            auto load_k = [&](int kt) {
                const int st = kt & 1;
                const uint32_t dst = base + kOffK + st * 2 * kKImg, bar = bar_k + 8 * st;
                mbar_expect_tx(bar, 2 * kKImg);
                bulk_g2s(dst, a.kh + (kv0 + kt) * kKImg, kKImg, bar);
                bulk_g2s(dst + kKImg, a.kl + (kv0 + kt) * kKImg, kKImg, bar);
            };
            constexpr uint32_t idS = idesc_bf16_f32(kPfRows, kPfKeys);
            const size_t qi = ((size_t)b * a.Hq + j) * a.nqt + qt;
            mbar_expect_tx(bar_q, 2 * kQImg);
            bulk_g2s(base + kOffQh, a.qh + qi * kQImg, kQImg, bar_q);
            bulk_g2s(base + kOffQl, a.ql + qi * kQImg, kQImg, bar_q);
            for (int kt = 0; kt < min(nkv, 2); ++kt) load_k(kt);
            ok = mbar_wait(q_tm, 0);  // Q hi and lo are in tensor memory
#pragma unroll 1
            for (int kt = 0; kt < nkv && ok; ++kt) {
                const int bb = kt & 1;
                const uint32_t ph = (kt >> 1) & 1;
                if (kt >= 2) ok = mbar_wait(s_free + 8 * bb, ph ^ 1u);  // the softmax has read S(kt - 2)
                ok = ok && mbar_wait(bar_k + 8 * bb, ph);
                if (!ok) break;
                tc_fence_after();
                // S of tile kt into buffer bb: Qh Kh^T + Ql Kh^T + Qh Kl^T over the 128 dims
                const uint32_t ks = base + kOffK + bb * 2 * kKImg, dS = tmem + 64 * bb;
                // the 24 MMAs issued back to back (one thread issues one MMA per ~50 cycles
                // only when nothing else sits between them): descriptors of the k-steps are
                // the stage's base descriptor plus the step's offset in 16-byte units
                const uint64_t dkh0 = sw128_desc(ks), dkl0 = sw128_desc(ks + kKImg);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint32_t ko = ((k >> 2) * (kKImg / 2) + (k & 3) * 32) >> 4;
                    mma_bf16_ts(dS, tmem + kTmQh + 8 * k, dkh0 + ko, idS, k > 0);
                    mma_bf16_ts(dS, tmem + kTmQl + 8 * k, dkh0 + ko, idS, 1);
                    mma_bf16_ts(dS, tmem + kTmQh + 8 * k, dkl0 + ko, idS, 1);
                }
                mma_commit(s_full + 8 * bb);
                if (kt + 2 < nkv) {  // S(kt) has read key stage bb: refill it
                    ok = mbar_wait(s_full + 8 * bb, ph);
                    if (ok) load_k(kt + 2);
                }
            }
            if (!ok) atomicOr(a.err, HSQ_DEVERR_WAIT);
        } else if (warp == kPfSoftThreads / 32 + 1 && lanei == 0) {
            auto load_v = [&](int kt) {
                const int st = kt & 1;
                mbar_expect_tx(bar_v + 8 * st, kVImg);
                bulk_g2s(base + kOffV + st * kVImg, a.vt + (kv0 + kt) * kVImg, kVImg, bar_v + 8 * st);
            };
            constexpr uint32_t idO = idesc_bf16_f32(kPfRows, kDim);
            for (int kt = 0; kt < min(nkv, 2); ++kt) load_v(kt);
#pragma unroll 1
            for (int kt = 0; kt < nkv && ok; ++kt) {
                const int bb = kt & 1;
                const uint32_t ph = (kt >> 1) & 1;
                ok = mbar_wait(p_full + 8 * bb, ph) && mbar_wait(bar_v + 8 * bb, ph);
                if (!ok) break;
                tc_fence_after();
                // O_k += Ph_k V_k + Pl_k V_k for key half k (keys 32 k .. + 31: two slices of 16)
                const uint32_t vs = base + kOffV + bb * kVImg, pb = base + kOffP + bb * 2 * kPImg;
                const uint64_t dv0 = sw128_desc(vs), dph0 = sw128_desc(pb), dpl0 = sw128_desc(pb + kPImg);
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        const uint32_t o = ((2 * hf + k) * 32) >> 4;
                        mma_bf16(tmem + 128 + 128 * hf, dph0 + o, dv0 + o, idO, (kt > 0) | (k > 0));
                        mma_bf16(tmem + 128 + 128 * hf, dpl0 + o, dv0 + o, idO, 1);
                    }
                }
                mma_commit(o_done + 8 * bb);
                if (kt + 2 < nkv) {  // P V of tile kt has read value stage bb: refill it
                    ok = mbar_wait(o_done + 8 * bb, ph);
                    if (ok) load_v(kt + 2);
                }
            }
            if (!ok) atomicOr(a.err, HSQ_DEVERR_WAIT);
        }
    } else {
        // ---- softmax: 8 warps, query row = TMEM lane, key half = warp >> 2 ----
        const int quarter = warp & 3, half = warp >> 2;
        const int row = 32 * quarter + lanei;
        const uint32_t lanes = (uint32_t)(32 * quarter) << 16;
        const uint32_t tO = tmem + lanes + 128 + 128 * half;
        const int t = qt * kPfRows + row;
        {   // Q (hi: warps 0-3, lo: warps 4-7) from its shared-memory image into tensor memory,
            // row = lane, dims in pairs along the columns
            ok = mbar_wait(bar_q, 0);
            if (!ok) atomicOr(a.err, HSQ_DEVERR_WAIT);  // (arrives all the same: no one waits forever)
            const uint8_t* img = gbase + (half ? kOffQl : kOffQh) + row * 128;
            float w[32];
#pragma unroll
            for (int blk = 0; blk < 2 && ok; ++blk) {
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 v = *reinterpret_cast<const uint4*>(img + blk * (kQImg / 2) + ((c ^ (row & 7)) << 4));
                    w[4 * c] = __uint_as_float(v.x);
                    w[4 * c + 1] = __uint_as_float(v.y);
                    w[4 * c + 2] = __uint_as_float(v.z);
                    w[4 * c + 3] = __uint_as_float(v.w);
                }
                tmem_st32(tmem + lanes + (half ? kTmQl : kTmQh) + 32 * blk, w);
            }
            tc_fence_before();
            mbar_arrive(q_tm);
        }
        float m_used = -INFINITY, lsum = 0.f;
#pragma unroll 1
        for (int kt = 0; kt < nkv; ++kt) {
            const int bb = kt & 1;
            const uint32_t ph = (kt >> 1) & 1;
            ok = mbar_wait(s_full + 8 * bb, ph);
            if (!ok) break;
            tc_fence_after();
            float x[32];
            tmem_ld32(tmem + lanes + 64 * bb + 32 * half, x);
            tc_fence_before();
            mbar_arrive(s_free + 8 * bb);
            // (the queries carry the log2-domain softmax scale; only the two diagonal
            // tiles have keys after some of the tile's queries)
            float mt = -INFINITY;
            if (kt >= nkv - 2) {
                const int key0 = kt * kPfKeys + 32 * half;
#pragma unroll
                for (int c = 0; c < 32; ++c) x[c] = key0 + c <= t ? x[c] : -INFINITY;
            }
#pragma unroll
            for (int c = 0; c < 32; ++c) mt = fmaxf(mt, x[c]);
            const float m_new = fmaxf(m_used, mt);
            const bool raise = m_new > m_used + 8.f;  // (the half's first unmasked key raises it from -inf)
            const float alpha = raise ? (m_used == -INFINITY ? 0.f : ex2_approx(m_used - m_new)) : 1.f;
            if (raise) {
                lsum *= alpha;
                m_used = m_new;
            }
            if (kt > 0 && __any_sync(0xffffffffu, raise)) {  // rescale this half's O row: P V of tile kt - 1 first
                ok = mbar_wait(o_done + 8 * (bb ^ 1), ((kt - 1) >> 1) & 1);
                if (!ok) break;
                tc_fence_after();
#pragma unroll 1
                for (int c0 = 0; c0 < kDim; c0 += 32) {
                    float o[32];
                    tmem_ld32(tO + c0, o);
#pragma unroll
                    for (int c = 0; c < 32; ++c) o[c] *= alpha;
                    tmem_st32(tO + c0, o);
                }
            }
            if (kt >= 2) {  // P buffer bb: P V of tile kt - 2 has read it
                ok = mbar_wait(o_done + 8 * bb, ph ^ 1u);
                if (!ok) break;
            }
            const float m_eff = m_used == -INFINITY ? 0.f : m_used;  // (no key yet: every p is 0)
            float psum = 0.f;
            uint8_t* prow_h = gbase + kOffP + bb * 2 * kPImg + row * 128;
            uint8_t* prow_l = prow_h + kPImg;
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                uint32_t wh[4], wl[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float p0 = ex2_approx(x[8 * cc + 2 * e] - m_eff), p1 = ex2_approx(x[8 * cc + 2 * e + 1] - m_eff);
                    psum += p0 + p1;
                    const __nv_bfloat162 hp = __floats2bfloat162_rn(p0, p1);
                    const __nv_bfloat162 lp = __floats2bfloat162_rn(p0 - __low2float(hp), p1 - __high2float(hp));
                    wh[e] = *reinterpret_cast<const uint32_t*>(&hp);
                    wl[e] = *reinterpret_cast<const uint32_t*>(&lp);
                }
                const uint32_t off = (uint32_t)(((4 * half + cc) ^ (row & 7)) << 4);
                *reinterpret_cast<uint4*>(prow_h + off) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
                *reinterpret_cast<uint4*>(prow_l + off) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
            }
            lsum += psum;
            fence_async_smem();
            tc_fence_before();
            mbar_arrive(p_full + 8 * bb);
        }
        if (ok) ok = mbar_wait(o_done + 8 * ((nkv - 1) & 1), ((nkv - 1) >> 1) & 1);  // the last P V
        if (!ok) atomicOr(a.err, HSQ_DEVERR_WAIT);
        // the row's two halves: maxima and sums, then each thread writes output columns
        // 64 half .. + 63 from its own O there plus the other half's (through the key stages)
        named_bar_sync(1, kPfSoftThreads);
        float (*s_ml)[2][kPfRows] = reinterpret_cast<float (*)[2][kPfRows]>(gbase + kOffV);
        s_ml[half][0][row] = m_used;
        s_ml[half][1][row] = lsum;
        named_bar_sync(1, kPfSoftThreads);
        tc_fence_after();
        const float m_o = s_ml[half ^ 1][0][row], l_o = s_ml[half ^ 1][1][row];
        const float M = fmaxf(m_used, m_o);
        const float w_me = m_used == -INFINITY ? 0.f : ex2_approx(m_used - M);
        const float w_ot = m_o == -INFINITY ? 0.f : ex2_approx(m_o - M);
        const float L = lsum * w_me + l_o * w_ot;
        const float inv = L > 0.f ? 1.0f / L : 0.f;
        // [2 halves][64 columns][128 rows]: the 32 rows of a warp are consecutive words
        // for every column, so the stores and loads below are free of bank conflicts
        float* xch = reinterpret_cast<float*>(gbase + kOffK);
        float o[32];
#pragma unroll 1
        for (int c0 = 0; c0 < 64; c0 += 32) {
            tmem_ld32(tO + 64 * (half ^ 1) + c0, o);
#pragma unroll
            for (int c = 0; c < 32; ++c) xch[((half ^ 1) * 64 + c0 + c) * kPfRows + row] = o[c] * w_me;
        }
        named_bar_sync(1, kPfSoftThreads);
        float* orow = a.out + (((size_t)b * a.Hq + j) * a.T + (t < a.T ? t : 0)) * kDim + 64 * half;
#pragma unroll 1
        for (int c0 = 0; c0 < 64; c0 += 32) {
            tmem_ld32(tO + 64 * half + c0, o);
            if (t < a.T && ok) {
                const float* other = xch + ((size_t)half * 64 + c0) * kPfRows + row;
#pragma unroll
                for (int c = 0; c < 32; c += 4)
                    *reinterpret_cast<float4*>(orow + c0 + c) = make_float4(
                        (o[c] * w_me + other[c * kPfRows]) * inv, (o[c + 1] * w_me + other[(c + 1) * kPfRows]) * inv,
                        (o[c + 2] * w_me + other[(c + 2) * kPfRows]) * inv,
                        (o[c + 3] * w_me + other[(c + 3) * kPfRows]) * inv);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// Query operand images: RoPE at the query's position in fp32, times the
// softmax scale log2(e) / sqrt(d), split into bf16 hi + lo.  One CTA of 256
// threads per (128-row tile, query head, sequence); each half-warp handles 8
// rows.
__global__ void __launch_bounds__(256) prefill_q_kernel(const uint16_t* __restrict__ Q, uint8_t* qh, uint8_t* ql,
                                                        int Hq, int T, int nqt, Tables tb) {
    const int qt = blockIdx.x, j = blockIdx.y, b = blockIdx.z;
    const int hw = threadIdx.x >> 4, l = hlane();
    const size_t img = (((size_t)b * Hq + j) * nqt + qt) * kQImg;
#pragma unroll 1
    for (int r = hw; r < kPfRows; r += 16) {
        const int t = qt * kPfRows + r;
        float x[8];
        if (t < T) {
            load_bf16x8(Q + (((size_t)b * Hq + j) * T + t) * kDim, x);
            rope(x, t, tb);
#pragma unroll
            for (int i = 0; i < 8; ++i) x[i] *= kLogitScaleLog2;  // logits come out in the log2 domain
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) x[i] = 0.f;
        }
#pragma unroll
        for (int blk = 0; blk < 2; ++blk) {
            uint16_t hi[4], lo[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) split_bf16(x[4 * blk + k], hi[k], lo[k]);
            const uint32_t off = sw128_row_quad(kPfRows, r, blk, l);
            *reinterpret_cast<uint2*>(qh + img + off) =
                make_uint2((uint32_t)hi[0] | ((uint32_t)hi[1] << 16), (uint32_t)hi[2] | ((uint32_t)hi[3] << 16));
            *reinterpret_cast<uint2*>(ql + img + off) =
                make_uint2((uint32_t)lo[0] | ((uint32_t)lo[1] << 16), (uint32_t)lo[2] | ((uint32_t)lo[3] << 16));
        }
    }
}

// Key and value operand images without the encode (attention on its own):
// one CTA of 256 threads per (64-key tile, KV head, sequence); half-warps
// take the tile's keys (RoPE'd, split) and values (transposed) in turn.
__global__ void __launch_bounds__(256) prefill_kv_kernel(const uint16_t* __restrict__ K, const uint16_t* __restrict__ V,
                                                         uint8_t* kh, uint8_t* kl, uint8_t* vt, int Hkv, int T, int nkt,
                                                         Tables tb) {
    const int kt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int hw = threadIdx.x >> 4, l = hlane();
    const size_t img = (((size_t)b * Hkv + h) * nkt + kt) * kKImg;
#pragma unroll 1
    for (int r = hw; r < 2 * kPfKeys; r += 16) {
        const int row = r & (kPfKeys - 1), t = kt * kPfKeys + row;
        const bool val = r >= kPfKeys;
        float x[8];
        if (t < T) {
            load_bf16x8((val ? V : K) + (((size_t)b * Hkv + h) * T + t) * kDim, x);
            if (!val) rope(x, t, tb);
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) x[i] = 0.f;
        }
        if (!val) {
#pragma unroll
            for (int blk = 0; blk < 2; ++blk) {
                uint16_t hi[4], lo[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) split_bf16(x[4 * blk + k], hi[k], lo[k]);
                const uint32_t off = sw128_row_quad(kPfKeys, row, blk, l);
                *reinterpret_cast<uint2*>(kh + img + off) =
                    make_uint2((uint32_t)hi[0] | ((uint32_t)hi[1] << 16), (uint32_t)hi[2] | ((uint32_t)hi[3] << 16));
                *reinterpret_cast<uint2*>(kl + img + off) =
                    make_uint2((uint32_t)lo[0] | ((uint32_t)lo[1] << 16), (uint32_t)lo[2] | ((uint32_t)lo[3] << 16));
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int d = (i < 4 ? 4 * l : 64 + 4 * l) + (i & 3);
                *reinterpret_cast<uint16_t*>(vt + img + sw128_elem(d, row)) =
                    __bfloat16_as_ushort(__float2bfloat16_rn(x[i]));
            }
        }
    }
}

}  // namespace

namespace hsq {

PrefillImages prefill_images(void* ws, int B, int Hq, int Hkv, int T) {
    PrefillImages im{};
    im.nqt = (T + kPfRows - 1) / kPfRows;
    im.nkt = 2 * im.nqt;
    uint8_t* p = static_cast<uint8_t*>(ws);
    const size_t q = (size_t)B * Hq * im.nqt * kQImg, k = (size_t)B * Hkv * im.nkt * kKImg;
    im.qh = p;
    im.ql = p + q;
    im.kh = p + 2 * q;
    im.kl = p + 2 * q + k;
    im.vt = p + 2 * q + 2 * k;
    im.bytes = 2 * q + 3 * k;
    return im;
}

hsq_status prefill_prep_q(hsq_ctx* ctx, const PrefillImages& im, const void* Q, int B, int T, cudaStream_t st) {
    const dim3 grid(im.nqt, ctx->cfg.n_q_heads, B);
    prefill_q_kernel<<<grid, 256, 0, st>>>(static_cast<const uint16_t*>(Q), im.qh, im.ql, ctx->cfg.n_q_heads, T,
                                           im.nqt, make_tables(ctx));
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? HSQ_OK : cuda_fail(ctx, e, "prefill_q_kernel");
}

hsq_status prefill_prep_kv(hsq_ctx* ctx, const PrefillImages& im, const void* K, const void* V, int B, int T,
                           cudaStream_t st) {
    const dim3 grid(im.nkt, ctx->cfg.n_kv_heads, B);
    prefill_kv_kernel<<<grid, 256, 0, st>>>(static_cast<const uint16_t*>(K), static_cast<const uint16_t*>(V), im.kh,
                                            im.kl, im.vt, ctx->cfg.n_kv_heads, T, im.nkt, make_tables(ctx));
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? HSQ_OK : cuda_fail(ctx, e, "prefill_kv_kernel");
}

hsq_status prefill_attention(hsq_ctx* ctx, const PrefillImages& im, float* out, int B, int T, cudaStream_t st) {
    const void* fn = (const void*)prefill_attn_kernel;
    cudaError_t e = raise_smem_limit(fn, ctx->device, kPfSmem);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaFuncSetAttribute(prefill)");
    PrefillArgs a{im.qh, im.ql, im.kh, im.kl, im.vt, out, ctx->d_err, ctx->cfg.n_q_heads, ctx->cfg.n_kv_heads, T,
                  im.nqt, im.nkt};
    const dim3 grid(im.nqt, ctx->cfg.n_q_heads, B);
    prefill_attn_kernel<<<grid, kPfThreads, kPfSmem, st>>>(a);
    e = cudaGetLastError();
    return e == cudaSuccess ? HSQ_OK : cuda_fail(ctx, e, "prefill_attn_kernel");
}

}  // namespace hsq
