// The fused decode-step kernel (one thread-block cluster per (b, KV head))
// and its host-side launch plan.  Included once per head ratio by
// hsq_decode_r<R>.cu, which instantiates it for R (and both group sizes).
//
// Decode process: Tamarin (HSQ) technical summary (gist.science
// rs-10297225), section 2 (route against the L2 summaries, fetch and
// dequantise the selected L3 originals, re-rotate to position, attend over
// the union with the fetched summaries masked).
#pragma once

#include <algorithm>

#include "hsq_device.cuh"

namespace {

// ---------------------------------------------------------------------------
// Decode step: one thread-block cluster per (b, KV head).  grid = (S, B*Hkv),
// cluster = (S, 1, 1), 256 threads per CTA.  Split s owns a contiguous share
// of the L2 groups and of the L1 slots of its (b, h) and an even share of the
// selected records.  The splits of a (b, h) exchange data only through
// distributed shared memory, by pushing (remote stores), each exchange
// closed by one cluster barrier:
//   1. stage the split's L2 summaries, L1 tokens, the sequence's L1 bitmap,
//      the codebook and the RoPE angle rows it may need (cp.async);
//   2. rotate the query heads; per-head logits of the split's L2 groups and,
//      with kRoute, the routing score n_g * (sum_j q~_j) . c3[codes] (the
//      arithmetic of the routing kernel, so both select the same groups),
//      whose key is pushed into every split's copy of the score array;
//   3. kRoute: after one barrier every split holds all G keys and runs the
//      same block-wide top-beta (identical result in every split);
//      otherwise the caller's selection is validated and used;
//   4. gather this split's share of the selected L3 records (zero copy when
//      L3 is host memory) and, while they travel, add the L1 tokens and the
//      unselected non-empty summaries;
//   5. recovered tokens: dequantise, inverse WHT, RoPE at the token's
//      position (per-record base angle plus a small offset), logits against
//      the RoPE'd queries, values kept in the rotated frame;
//   6. the CTA's softmax partial of each query head, rotated back to the
//      original frame (a linear map, so it commutes with the merge), is pushed
//      in pieces: split r owns a slice of 4-dim quads of every head, merges the
//      S partials of its quads after the last barrier and stores them.
// Each half-warp runs its own online softmax over its entries, two entries
// per step.  Every loop has warp-uniform bounds (entries past the end are
// computed on a clamped index and masked), so all shuffles run on full
// warps.  kStaged: the split's L2 / L1 slices, the L1 bitmap row and the
// split's L2 logits live in shared memory; without it (contexts too long for
// shared memory) they are read in place from global memory and the L2
// logits are recomputed.
// ---------------------------------------------------------------------------

constexpr int kMaxSplits = 16;   // largest (non-portable) cluster

// Threads per CTA of the decode kernel.  8 warps: 12 warps (384 threads,
// which still fit the R <= 5 softmax state in registers) measured slower.
template <int R>
__host__ __device__ constexpr int dec_threads() { return 256; }
enum : int { kStageL2 = 1, kKeepLogits = 2, kStageL1 = 4, kStageBitmap = 8, kStageSketch = 16 };

struct DecodeArgs {
    const float* q; const int32_t* pos; int32_t* sel; float* out; int* err; int from_staging;
};

constexpr int kStagedFlags = kStageL2 | kKeepLogits | kStageL1 | kStageBitmap;

struct DecodeLayout {
    int span, l1span, nlev, nb0;
    unsigned l2k, l2v, l2kn, l2vn, cnt, l1k, l1v, l1kn, l1vn, logit, sel, mask, bitmap, l1qs, l1qn;
    unsigned lev, b0, off, base, rbits, inbox, rec, total;
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

// The output merge: split r of S owns the 4-dim quads [quad0(r), quad0(r + 1)) of every
// query head; each split pushes, per head, its partial's quads to their owners and its
// (max, sum) to every split.  Inbox row (head j, source split): the owner's quads, then
// max and sum (a stride of whole quads).
__host__ __device__ inline int quad0(int r, int S) { return (32 * r) / S; }
__host__ __device__ inline int inbox_stride(int S) { return 4 * ((32 + S - 1) / S + 1); }

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
    L.l2k = L.l2v = L.l2kn = L.l2vn = L.cnt = L.l1k = L.l1v = L.l1kn = L.l1vn = L.logit = L.bitmap = 0;
    L.l1qs = L.l1qn = 0;
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
    if (flags & kStageSketch) {  // TQ-QKV: the sketches of the split's L1 keys
        L.l1qs = (unsigned)o; o = al16(o + (size_t)L.l1span * 16);
        L.l1qn = (unsigned)o; o = al16(o + (size_t)L.l1span * 4);
    }
    if (flags & kKeepLogits) { L.logit = (unsigned)o; o = al16(o + (size_t)L.span * R * 4); }
    if (flags & kStageBitmap) { L.bitmap = (unsigned)o; o = al16(o + (size_t)((T + 31) / 32) * 4); }
    L.sel = (unsigned)o; o = al16(o + (size_t)beta * 4);
    L.mask = (unsigned)o; o = al16(o + (size_t)((L.span + 31) / 32) * 4);
    L.lev = (unsigned)o; o = al16(o + (size_t)L.nlev * 16 * row);
    L.b0 = (unsigned)o; o = al16(o + (size_t)L.nb0 * row);
    L.off = (unsigned)o; o = al16(o + (size_t)N * row);
    L.base = (unsigned)o; o = al16(o + (size_t)2 * kBatchRecs * row);   // two batches in flight
    L.rbits = (unsigned)o; o = al16(o + (size_t)2 * kBatchRecs * 4);
    L.inbox = (unsigned)o; o = al16(o + (size_t)R * S * inbox_stride(S) * 4);
    // one region, used in turn for: every split's routing keys (until the
    // selection is made), two batches of gathered L3 records, the warp partials
    size_t rec = 2 * (size_t)kFetchBatchBytes;
    const size_t merge = (size_t)(dec_threads<R>() / 32) * R * hsq::kPartStride * 4;
    if (merge > rec) rec = merge;
    if (route && (size_t)G * 4 > rec) rec = (size_t)G * 4;
    L.rec = (unsigned)o; o = al16(o + rec);
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
            // rescale by selects, not a branch (the two half-warps of a warp diverge here)
            const float a = oka ? xa[j] : -INFINITY, b = okb ? xb[j] : -INFINITY;
            const float mn = fmaxf(m[j], fmaxf(a, b));
            const float corr = mn > m[j] ? fast_exp2(m[j] - mn) : 1.f;
            l[j] *= corr;
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[j][i] *= corr;
            m[j] = mn;
            const float pa = oka ? fast_exp2(a - mn) : 0.f;
            const float pb = okb ? fast_exp2(b - mn) : 0.f;
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

// Walsh-Hadamard transform of 128 values held 4 per lane (dims 4 lane .. 4 lane + 3)
// across a full warp: index bits 0-1 in registers, bits 2-6 across the lanes
__device__ __forceinline__ void fwht_quad(float4& v) {
    const float a = v.x + v.y, b = v.x - v.y, c = v.z + v.w, d = v.z - v.w;
    v = make_float4(a + c, b + d, a - c, b - d);
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
        const float sgn = (lane & m) ? -1.f : 1.f;  // upper lane: p - v, lower lane: v + p
        v.x = fmaf(sgn, v.x, __shfl_xor_sync(0xffffffffu, v.x, m));
        v.y = fmaf(sgn, v.y, __shfl_xor_sync(0xffffffffu, v.y, m));
        v.z = fmaf(sgn, v.z, __shfl_xor_sync(0xffffffffu, v.z, m));
        v.w = fmaf(sgn, v.w, __shfl_xor_sync(0xffffffffu, v.w, m));
    }
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}

// The 2R logits of a pair in every lane: xa[j] = scale * (q_j . ka), xb likewise.
// xs: this half-warp's 16-float scratch in shared memory.
template <int R>
__device__ __forceinline__ void pair_logits(const float (&q)[R][8], const float (&ka)[8], const float (&kb)[8],
                                            float scale, float* xs, float (&xa)[R], float (&xb)[R]) {
    int idx;
    const float d = pair_dots<R>(q, ka, kb, idx);
    __syncwarp();  // the previous pair's reads are done
    if (idx < 2 * R) xs[idx] = d * scale;
    __syncwarp();
#pragma unroll
    for (int j = 0; j < R; ++j) {
        xa[j] = xs[j];
        xb[j] = xs[R + j];
    }
}

// pair_logits plus the residual-sketch terms of TQ-QKV:
// xa[j] = scale * (q_j . ka + sq_j . ca), sq_j = S Pi q^r_j, ca the signed sketch of a.
template <int R>
__device__ __forceinline__ void pair_logits_qjl(const float (&q)[R][8], const float (&ka)[8], const float (&kb)[8],
                                                const float (&sq)[R][8], const float (&ca)[8], const float (&cb)[8],
                                                float scale, float* xs, float (&xa)[R], float (&xb)[R]) {
    int idx;
    const float d = pair_dots2<R>(q, ka, kb, sq, ca, cb, idx);
    __syncwarp();  // the previous pair's reads are done
    if (idx < 2 * R) xs[idx] = d * scale;
    __syncwarp();
#pragma unroll
    for (int j = 0; j < R; ++j) {
        xa[j] = xs[j];
        xb[j] = xs[R + j];
    }
}

__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;\n" ::: "memory");
}

__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.aligned;\n" ::: "memory");
}

// kRot: TurboQuant (rotated frame); false: Plain-KV (identity, no signs).
// kQJL: TQ-QKV, the logits of L1 and fetched tokens carry the residual-sketch term.
// kHot: the hot-group table -- a selected group whose slot g & hot_mask is
// tagged g is read from the device copy instead of L3; a group fetched from L3
// is copied into its slot, and tagged, when it is the only selected group of
// this step mapping there (so a step never reads and writes one slot; every
// slot is written by the one CTA that fetched its record).  Tags are staged
// before the cluster barrier that precedes selection, so no CTA writes a tag
// that another CTA of the cluster is still staging.
template <int R, int N, bool kRoute, bool kStaged, bool kRot, bool kQJL = false, bool kHot = false>
__global__ void __launch_bounds__(dec_threads<R>(), 1) decode_kernel(CacheView c, DecodeArgs a, Tables tb) {
    namespace cgx = cooperative_groups;
    constexpr int NT = dec_threads<R>(), NH = NT / 16, NW = NT / 32;
    constexpr int kChunksPT = (kFetchBatchBytes / 16 + NT - 1) / NT;  // gathered 16-B chunks per thread
    extern __shared__ __align__(16) uint8_t s_dyn[];
    __shared__ __align__(16) float s_cb[hsq::kCodebookFloats];
    __shared__ __align__(16) float s_qt[R][kDim];
    __shared__ __align__(16) float s_qr[R][kDim];
    __shared__ __align__(16) float s_sq[kQJL ? R : 1][kDim];  // S Pi q^r_j (TQ-QKV)
    // TQ-QKV: the sketch words and norms of a batch's fetched tokens, gathered with its records
    __shared__ __align__(16) uint4 s_tsk[kQJL ? 2 : 1][kQJL ? kFetchBatchBytes / 136 : 1];
    __shared__ float s_tnm[kQJL ? 2 : 1][kQJL ? kFetchBatchBytes / 136 : 1];
    __shared__ __align__(16) float s_x[NH][16];
    __shared__ SelectSmem s_ss;
    __shared__ __align__(16) uint32_t s_stats[kMaxSplits][4];  // per split: non-empty keys, max key, min key
    static_assert(!kHot || kRoute, "the hot-group table belongs to the fused (routing) step");
    constexpr int kHotSlots = kHot ? hsq::kMaxHotSlots : 32;
    __shared__ __align__(16) int32_t s_htag[kHot ? hsq::kMaxHotSlots : 4];  // the table's tags at launch
    __shared__ uint32_t s_hone[kHotSlots / 32], s_htwo[kHotSlots / 32];   // slots selected once / again

    constexpr int RB = N * 136;
    constexpr int kBatchRecs = kFetchBatchBytes / RB;
    constexpr int kRecChunks = RB / 16;

    // first phase of the cluster barrier: every CTA of the cluster has started
    // (completed by cluster_wait before the first remote store)
    cluster_arrive_relaxed();
    cgx::cluster_group cluster = cgx::this_cluster();
    const int S = (int)cluster.num_blocks();
    const int s = (int)cluster.block_rank();
    const int bh = blockIdx.y, b = bh / c.Hkv, h = bh % c.Hkv;
    // tier buffers of this head: bh, except under per-query-head routing (run with R = 1)
    const size_t bb = R == 1 ? buf_head(c, b, h) : (size_t)bh;
    const int tid = threadIdx.x, hw = tid >> 4, l = hlane(), lane = tid & 31, warp = tid >> 5;
    // Under a programmatic (overlapped) launch: wait for the stream's preceding
    // kernel to complete before touching global memory, then let the next one be
    // scheduled.  Both are no-ops under ordinary stream order.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    constexpr int fl = kStaged ? (kStagedFlags | (kQJL ? kStageSketch : 0)) : 0;
    const DecodeLayout L = decode_layout<R, N>(c.G, c.cap, S, c.max_l1, c.beta, kRoute, fl);

    const int g0 = (int)((long long)c.G * s / S), g1 = (int)((long long)c.G * (s + 1) / S);
    const int n2 = g1 - g0;
    const int cnt1 = min(__ldg(c.l1_count + b), c.max_l1);
    const int e0 = (int)((long long)cnt1 * s / S), e1 = (int)((long long)cnt1 * (s + 1) / S);
    const int n1 = e1 - e0;
    const int f0 = (int)((long long)c.beta * s / S), f1 = (int)((long long)c.beta * (s + 1) / S);
    const int nfetch = f1 - f0;

    // inputs: staged copies in shared memory, or read in place
    const uint8_t* g_l2k = c.l2_kc + (bb * c.G + g0) * 48;
    const uint8_t* g_l2v = c.l2_vc + (bb * c.G + g0) * 48;
    const float* g_l2kn = c.l2_kn + bb * c.G + g0;
    const float* g_l2vn = c.l2_vn + bb * c.G + g0;
    const uint8_t* g_cnt = c.l2_cnt + (size_t)b * c.G + g0;
    const uint8_t* g_l1k = c.l1_kc + (bb * c.max_l1 + e0) * 64;
    const uint8_t* g_l1v = c.l1_vc + (bb * c.max_l1 + e0) * 64;
    const float* g_l1kn = c.l1_kn + bb * c.max_l1 + e0;
    const float* g_l1vn = c.l1_vn + bb * c.max_l1 + e0;
    const uint32_t* g_bitmap = c.l1_bitmap + (size_t)b * c.W;
    constexpr bool st2 = kStaged, st1 = kStaged, stb = kStaged, keep = kStaged;
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
    int* s_sel = reinterpret_cast<int*>(s_dyn + L.sel);
    uint32_t* s_mask = reinterpret_cast<uint32_t*>(s_dyn + L.mask);
    float* s_lev = reinterpret_cast<float*>(s_dyn + L.lev);
    float* s_b0 = reinterpret_cast<float*>(s_dyn + L.b0);
    float* s_off = reinterpret_cast<float*>(s_dyn + L.off);
    float* s_base = reinterpret_cast<float*>(s_dyn + L.base);
    uint32_t* s_rbits = reinterpret_cast<uint32_t*>(s_dyn + L.rbits);
    float* s_inbox = reinterpret_cast<float*>(s_dyn + L.inbox);
    uint8_t* s_rec = s_dyn + L.rec;
    uint32_t* s_all = reinterpret_cast<uint32_t*>(s_dyn + L.rec);  // routing keys of all splits
    float* xs = &s_x[hw][0];

    // 0. the few values read straight into registers, issued before anything
    //    waits on them: position, this half-warp's query head, signs, counts
    const int pos_raw = __ldcg(a.pos + b);  // (q, pos, sel, out may be host-mapped)
    float qx[8];  // (only the R half-warps of the heads read; the rest compute on zeros)
    if (hw < R) {
        load_f32x8_cg(a.q + ((size_t)b * c.Hq + h * R + hw) * kDim, qx);
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) qx[i] = 0.f;
    }
    float sg[8];
    if constexpr (kRot) {
        load_signs_global(sg, c.signs);
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) sg[i] = 1.f;
    }
    const uint8_t cnt0 = st2 && tid < n2 ? __ldg(g_cnt + tid) : (uint8_t)0;

    // 1. stage the device-resident inputs of this split: first what the L2
    //    pass needs (one cp.async group), then the rest (a second group)
    if constexpr (st2) {
        stage16(s_dyn + L.l2k, g_l2k, n2 * 48);
        stage4(reinterpret_cast<float*>(s_dyn + L.l2kn), g_l2kn, n2);
    }
    if (tid < hsq::kCodebookFloats / 4) cp_async16(s_cb + 4 * tid, tb.cb + 4 * tid);
    cp_async_commit();
    if constexpr (st2) {
        stage16(s_dyn + L.l2v, g_l2v, n2 * 48);
        stage4(reinterpret_cast<float*>(s_dyn + L.l2vn), g_l2vn, n2);
    }
    if constexpr (st1) {
        stage16(s_dyn + L.l1k, g_l1k, n1 * 64);
        stage16(s_dyn + L.l1v, g_l1v, n1 * 64);
        stage4(reinterpret_cast<float*>(s_dyn + L.l1kn), g_l1kn, n1);
        stage4(reinterpret_cast<float*>(s_dyn + L.l1vn), g_l1vn, n1);
    }
    if constexpr (stb) stage4(reinterpret_cast<float*>(s_dyn + L.bitmap), reinterpret_cast<const float*>(g_bitmap), c.W);
    if constexpr (kQJL && st1) {
        stage16(s_dyn + L.l1qs, c.l1_qs + (bb * c.max_l1 + e0) * 4, n1 * 16);
        stage4(reinterpret_cast<float*>(s_dyn + L.l1qn), c.l1_qn + bb * c.max_l1 + e0, n1);
    }
    // RoPE rows: level k row j = hi[j * 16^k] (angle 256 j 16^k omega), b0 row j = lo[N j], off row n = lo[n]
    const int n_hi = (tb.max_pos + 255) / 256;
#pragma unroll 1
    for (int i = tid; i < L.nlev * 16 * 32; i += NT) {
        const int rowi = i >> 5, k = rowi >> 4, j = rowi & 15;
        const int src = j << (4 * k);
        if (src < n_hi) cp_async16(s_lev + 4 * i, tb.rope_hi + (size_t)src * kDim + 4 * (i & 31));
    }
#pragma unroll 1
    for (int i = tid; i < L.nb0 * 32; i += NT)
        cp_async16(s_b0 + 4 * i, tb.rope_lo + (size_t)(N * (i >> 5)) * kDim + 4 * (i & 31));
    stage16(s_off, tb.rope_lo, N * kDim * 4);
    if constexpr (kHot) stage16(s_htag, c.hot_tag + bb * (c.hot_mask + 1), (c.hot_mask + 1) * 4);
    cp_async_commit();
    for (int i = tid; i < (L.span + 31) / 32; i += NT) s_mask[i] = 0u;
    if constexpr (kHot) {
        for (int i = tid; i < kHotSlots / 32; i += NT) s_hone[i] = s_htwo[i] = 0u;
    }
    if constexpr (st2) {
        if (tid < n2) s_dyn[L.cnt + tid] = cnt0;
#pragma unroll 1
        for (int i = tid + NT; i < n2; i += NT) s_dyn[L.cnt + i] = __ldg(g_cnt + i);
    }

    // 2. query heads of this KV head: RoPE'd (original frame) and rotated
    const int pos = checked_pos(pos_raw, tb, a.err);
    prepare_queries<R>(qx, pos, sg, tb, s_qt, s_qr, kRot);
    cp_async_wait_group<1>();  // the L2 pass's inputs
    __syncthreads();
    // TQ-QKV: rows [i0, i1) of the sketched rotated queries S q~_j, 16 threads per row (8
    // dims each, a fixed half-warp reduction), every head; with `push` each row goes to
    // every split of the cluster (remote stores), else to this CTA's s_sq only
    auto sq_rows = [&](int i0, int i1, bool push) {
        const unsigned hm = half_mask();
#pragma unroll 1
        for (int i = i0 + hw; i < i1; i += NH) {
            const float4* srow = reinterpret_cast<const float4*>(c.qjl_s + (size_t)i * kDim) + 2 * l;
            const float4 s0 = __ldg(srow), s1 = __ldg(srow + 1);
            float v[R];
#pragma unroll
            for (int j = 0; j < R; ++j) {
                const float* qj = s_qt[j] + 8 * l;
                float a = s0.x * qj[0];
                a = fmaf(s0.y, qj[1], a); a = fmaf(s0.z, qj[2], a); a = fmaf(s0.w, qj[3], a);
                a = fmaf(s1.x, qj[4], a); a = fmaf(s1.y, qj[5], a); a = fmaf(s1.z, qj[6], a); a = fmaf(s1.w, qj[7], a);
                v[j] = half_sum(a, hm);
            }
            if (push) {
                if (l < S) {
#pragma unroll
                    for (int j = 0; j < R; ++j) *cluster.map_shared_rank(&s_sq[j][i], l) = v[j];
                }
            } else if (l == 0) {
#pragma unroll
                for (int j = 0; j < R; ++j) s_sq[j][i] = v[j];
            }
        }
    };
    if constexpr (kQJL && !kRoute) sq_rows(0, kDim, false);  // (read after the barriers that precede the L1 pass)

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
    if (kRoute) cluster_wait();  // every CTA of the cluster runs: remote stores may start
    if constexpr (kQJL && kRoute) sq_rows(kDim * s / S, kDim * (s + 1) / S, true);  // (in every split after the selection barrier)
    if constexpr (kRoute || keep) {
        // routing keys (each goes to every split, and so do this split's key
        // statistics) and the L2 logits per query head, one pass
        float gq[8];
        if constexpr (kRoute) {
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
        uint32_t* dst = kRoute && l < S ? cluster.map_shared_rank(s_all, l) + g0 : nullptr;
        int cn = 0;
        uint32_t mx = 0u, mn = 0xFFFFFFFFu;
#pragma unroll 1
        for (int blk = 0; blk < n2; blk += 2 * NH) {
            const int ia = blk + hw, ib = ia + NH;
            const int ja = min(ia, n2 - 1), jb = min(ib, n2 - 1);
            float va[8], vb[8];
            unpack3_smem(p_l2k + ja * 48, c3, 1.0f, va);
            unpack3_smem(p_l2k + jb * 48, c3, 1.0f, vb);
            if constexpr (kRoute) {
                float sa, sb;
                route_pair(gq, va, vb, sa, sb);
                // (flags are bitwise: no branch around the loads)
                const uint32_t ka = ((ia < n2) & (p_cnt[ja] > 0)) ? ordered_key(p_l2kn[ja] * sa) : 0u;
                const uint32_t kb = ((ib < n2) & (p_cnt[jb] > 0)) ? ordered_key(p_l2kn[jb] * sb) : 0u;
                if (dst && ia < n2) dst[ia] = ka;  // lane l < S writes this pair's keys into split l
                if (dst && ib < n2) dst[ib] = kb;
                const bool l0 = l == 0;
                cn += l0 ? (ka != 0u) + (kb != 0u) : 0;
                mx = max(mx, l0 ? max(ka, kb) : 0u);
                mn = min(mn, l0 ? min(ka ? ka : 0xFFFFFFFFu, kb ? kb : 0xFFFFFFFFu) : 0xFFFFFFFFu);
            }
            if constexpr (keep) {
                int idx;
                const float d = pair_dots<R>(qt, va, vb, idx);
                const bool first = idx < R;
                const int e = first ? ia : ib;
                const float kn = first ? p_l2kn[ja] : p_l2kn[jb];
                if ((idx < 2 * R) & (e < n2)) s_logit[e * R + (first ? idx : idx - R)] = kn * d * kLogitScaleLog2;
            }
        }
        if constexpr (kRoute) {
            cn = __reduce_add_sync(kFull, cn);
            mx = __reduce_max_sync(kFull, mx);
            mn = __reduce_min_sync(kFull, mn);
            if (lane == 0) { s_ss.red[0][warp] = (uint32_t)cn; s_ss.red[1][warp] = mx; s_ss.red[2][warp] = mn; }
            __syncthreads();
            if (tid < S) {
                uint32_t t = 0u, hx = 0u, lx = 0xFFFFFFFFu;
#pragma unroll
                for (int w = 0; w < NW; ++w) {
                    t += s_ss.red[0][w];
                    hx = max(hx, s_ss.red[1][w]);
                    lx = min(lx, s_ss.red[2][w]);
                }
                *reinterpret_cast<uint4*>(cluster.map_shared_rank(&s_stats[s][0], tid)) = make_uint4(t, hx, lx, 0u);
            }
        }
    }

    // 3. the selection of this (b, h)
    cp_async_wait_group<0>();  // everything staged (visible after the next barrier)
    if (kRoute) {
        cluster.sync();  // every split's keys and statistics are in every split
        select_top_beta<NT>(s_all, c.G, c.beta, s_sel, s_ss, &s_stats[0][0], S);
        __syncthreads();
        if (s == 0)
            for (int i = tid; i < c.beta; i += NT) a.sel[(size_t)bh * c.beta + i] = s_sel[i];
    } else {
        for (int i = tid; i < c.beta; i += NT) s_sel[i] = valid_sel(a.sel + (size_t)bh * c.beta, i, c.G, a.err);
        __syncthreads();
    }
    for (int i = tid; i < c.beta; i += NT) {
        const int g = s_sel[i];
        if (g >= g0 && g < g1) atomicOr(&s_mask[(g - g0) >> 5], 1u << ((g - g0) & 31));
        if constexpr (kHot) {
            if (g >= 0) {
                const int sl = g & c.hot_mask;
                const uint32_t bit = 1u << (sl & 31);
                if (atomicOr(&s_hone[sl >> 5], bit) & bit) atomicOr(&s_htwo[sl >> 5], bit);
            }
        }
    }

    // 4. gather this split's records (batch k: records f0 + k B .., loaded into
    //    registers one batch ahead -- zero-copy loads from host memory -- and
    //    stored to buffer k & 1 when consumed); meanwhile the L1 tokens and the
    //    unselected summaries.  Per record, its base angle g N omega (staged
    //    rows only) and its L1 bits go to slot k & 1.
    uint4 pre[kChunksPT];
    // TQ-QKV: thread u < kBatchRecs * N also gathers token u of the batch's records:
    // its sketch words and norm (norm 0 for a slot that is no token)
    uint4 psk = make_uint4(0u, 0u, 0u, 0u);
    float pnm = 0.f;
    auto issue = [&](int k) {
        const int r0 = f0 + k * kBatchRecs;
        const int nrec = min(kBatchRecs, f1 - r0);
        if constexpr (kQJL) {
            psk = make_uint4(0u, 0u, 0u, 0u);
            pnm = 0.f;
            if (tid < nrec * N) {
                const int rec = tid / N, n = tid - rec * N;
                const int g = s_sel[r0 + rec];
                const int t = g * N + n;
                if ((g >= 0) & (t < c.T)) {
                    const size_t ti = bb * (size_t)c.G * N + (size_t)t;
                    psk = __ldg(reinterpret_cast<const uint4*>(c.l3_qs) + ti);
                    pnm = __ldg(c.l3_qn + ti);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kChunksPT; ++u) {
            const int ch = tid + u * NT;
            pre[u] = make_uint4(0u, 0u, 0u, 0u);
            if (ch < nrec * kRecChunks) {
                const int rec = ch / kRecChunks, off = ch - rec * kRecChunks;
                const int i = r0 + rec;
                const int g = s_sel[i];
                if (g >= 0) {
                    const uint8_t* src = a.from_staging ? c.staging + ((size_t)bh * c.beta + i) * RB
                                                        : c.l3 + (bb * c.G + g) * RB;
                    if constexpr (kHot) {
                        const int sl = g & c.hot_mask;
                        if (s_htag[sl] == g) src = c.hot_rec + (bb * (c.hot_mask + 1) + sl) * RB;
                    }
                    pre[u] = __ldcg(reinterpret_cast<const uint4*>(src) + off);
                }
            }
        }
        if (hw < nrec) {
            const int g = s_sel[r0 + hw];
            if (g >= 0) {
                const int p0 = g * N;
                const float* br = s_b0 + ((p0 & 255) / N) * kDim;
                float4 cs = *reinterpret_cast<const float4*>(br + 4 * l);
                float4 sn = *reinterpret_cast<const float4*>(br + 64 + 4 * l);
#pragma unroll 1
                for (int k2 = 0; k2 < L.nlev; ++k2) {  // one 4-bit digit of p0 >> 8 per level
                    const int j = (p0 >> (8 + 4 * k2)) & 15;
                    if (j) {
                        const float* lr = s_lev + (k2 * 16 + j) * kDim;
                        angle_add4(cs, sn, *reinterpret_cast<const float4*>(lr + 4 * l),
                                   *reinterpret_cast<const float4*>(lr + 64 + 4 * l));
                    }
                }
                float* sb = s_base + ((k & 1) * kBatchRecs + hw) * kDim;
                *reinterpret_cast<float4*>(sb + 4 * l) = cs;
                *reinterpret_cast<float4*>(sb + 64 + 4 * l) = sn;
                if (l == 0)
                    s_rbits[(k & 1) * kBatchRecs + hw] =
                        (p_bitmap[p0 >> 5] >> (p0 & 31)) & ((N == 32) ? 0xFFFFFFFFu : ((1u << N) - 1u));
            }
        }
    };
    const int nbatch = (nfetch + kBatchRecs - 1) / kBatchRecs;
    issue(0);

    __syncthreads();  // s_mask complete

    Softmax<R> sm;
    sm.init();
    float sq[kQJL ? R : 1][8];  // this lane's coordinates of S q~_j (TQ-QKV)
    if constexpr (kQJL) {
#pragma unroll
        for (int j = 0; j < R; ++j) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                sq[j][k] = s_sq[j][4 * l + k];
                sq[j][4 + k] = s_sq[j][64 + 4 * l + k];
            }
        }
    }
    // TQ-QKV: the sketch words of a pair of L1 entries, loaded one step ahead
    uint4 nwa = make_uint4(0, 0, 0, 0), nwb = nwa;
    float nga = 0.f, ngb = 0.f;
    auto l1_sketch = [&](int blk_) {
        const int ja_ = min(blk_ + hw, n1 - 1), jb_ = min(blk_ + hw + NH, n1 - 1);
        if constexpr (st1) {  // staged with the split's other L1 inputs
            const uint4* qs = reinterpret_cast<const uint4*>(s_dyn + L.l1qs);
            const float* qn = reinterpret_cast<const float*>(s_dyn + L.l1qn);
            nwa = qs[ja_]; nwb = qs[jb_]; nga = qn[ja_]; ngb = qn[jb_];
        } else {
            const size_t ia = bb * c.max_l1 + e0 + ja_, ib = bb * c.max_l1 + e0 + jb_;
            nwa = __ldg(reinterpret_cast<const uint4*>(c.l1_qs) + ia);
            nwb = __ldg(reinterpret_cast<const uint4*>(c.l1_qs) + ib);
            nga = __ldg(c.l1_qn + ia);
            ngb = __ldg(c.l1_qn + ib);
        }
    };
    if constexpr (kQJL) {
        if (n1 > 0) l1_sketch(0);
    }
#pragma unroll 1
    for (int blk = 0; blk < n1; blk += 2 * NH) {
        const int ea = blk + hw, eb = ea + NH;
        const int ja = min(ea, n1 - 1), jb = min(eb, n1 - 1);
        float ka[8], kb[8], va[8], vb[8], xa[R], xb[R];
        const uint16_t* kra = reinterpret_cast<const uint16_t*>(p_l1k + ja * 64);
        const uint16_t* krb = reinterpret_cast<const uint16_t*>(p_l1k + jb * 64);
        const uint16_t* vra = reinterpret_cast<const uint16_t*>(p_l1v + ja * 64);
        const uint16_t* vrb = reinterpret_cast<const uint16_t*>(p_l1v + jb * 64);
        unpack4(kra[l], kra[16 + l], c4, p_l1kn[ja], ka);
        unpack4(krb[l], krb[16 + l], c4, p_l1kn[jb], kb);
        if constexpr (kQJL) {
            const uint4 wa = nwa, wb = nwb;
            const float ga = nga, gb = ngb;
            if (blk + 2 * NH < n1) l1_sketch(blk + 2 * NH);
            float ca[8], cb[8];
            sketch_signs(wa, kQjlScale * ga, ca);
            sketch_signs(wb, kQjlScale * gb, cb);
            pair_logits_qjl<R>(qt, ka, kb, sq, ca, cb, kLogitScaleLog2, xs, xa, xb);
        } else {
            pair_logits<R>(qt, ka, kb, kLogitScaleLog2, xs, xa, xb);
        }
        unpack4(vra[l], vra[16 + l], c4, p_l1vn[ja], va);
        unpack4(vrb[l], vrb[16 + l], c4, p_l1vn[jb], vb);
        sm.add2(xa, va, ea < n1, xb, vb, eb < n1);
    }
#pragma unroll 1
    for (int blk = 0; blk < n2; blk += 2 * NH) {
        const int ia = blk + hw, ib = ia + NH;
        const int ja = min(ia, n2 - 1), jb = min(ib, n2 - 1);
        const bool oka = (ia < n2) & (p_cnt[ja] > 0) & (((s_mask[ja >> 5] >> (ja & 31)) & 1u) == 0u);
        const bool okb = (ib < n2) & (p_cnt[jb] > 0) & (((s_mask[jb >> 5] >> (jb & 31)) & 1u) == 0u);
        if (!__any_sync(kFull, oka || okb)) continue;
        float va[8], vb[8], xa[R], xb[R];
        if constexpr (keep) {
#pragma unroll
            for (int j = 0; j < R; ++j) {
                xa[j] = s_logit[ja * R + j];
                xb[j] = s_logit[jb * R + j];
            }
        } else {
            float ka[8], kb[8];
            unpack3_smem(p_l2k + ja * 48, c3, p_l2kn[ja], ka);
            unpack3_smem(p_l2k + jb * 48, c3, p_l2kn[jb], kb);
            pair_logits<R>(qt, ka, kb, kLogitScaleLog2, xs, xa, xb);
        }
        unpack3_smem(p_l2v + ja * 48, c3, p_l2vn[ja], va);
        unpack3_smem(p_l2v + jb * 48, c3, p_l2vn[jb], vb);
        sm.add2(xa, va, oka, xb, vb, okb);
    }

    // 5. recovered tokens of the selected groups
    {
        float qr[R][8];
#pragma unroll
        for (int j = 0; j < R; ++j) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                qr[j][k] = s_qr[j][4 * l + k];
                qr[j][4 + k] = s_qr[j][64 + 4 * l + k];
            }
        }
#pragma unroll 1
        for (int kb_ = 0; kb_ < nbatch; ++kb_) {
            {   // batch kb_ lands in buffer kb_ & 1 (the loads were issued one batch ahead)
                uint4* dstb = reinterpret_cast<uint4*>(s_rec + (kb_ & 1) * kFetchBatchBytes);
#pragma unroll
                for (int u = 0; u < kChunksPT; ++u) {
                    const int ch = tid + u * NT;
                    if (ch < kFetchBatchBytes / 16) dstb[ch] = pre[u];
                }
                if constexpr (kQJL) {
                    if (tid < kBatchRecs * N) {
                        s_tsk[kb_ & 1][tid] = psk;
                        s_tnm[kb_ & 1][tid] = pnm;
                    }
                }
                if constexpr (kHot) {  // records fetched from L3 into their free slots
                    const int hr0 = f0 + kb_ * kBatchRecs;
                    const int hnb = min(kBatchRecs, f1 - hr0);
#pragma unroll
                    for (int u = 0; u < kChunksPT; ++u) {
                        const int ch = tid + u * NT;
                        if (ch < hnb * kRecChunks) {
                            const int rec = ch / kRecChunks, off = ch - rec * kRecChunks;
                            const int g = s_sel[hr0 + rec];
                            const int sl = g & c.hot_mask;
                            const uint32_t bit = 1u << (sl & 31);
                            const bool once = ((s_hone[sl >> 5] & ~s_htwo[sl >> 5]) & bit) != 0u;
                            if ((g >= 0) & once & (s_htag[sl] != g)) {
                                const size_t slot = bb * (c.hot_mask + 1) + sl;
                                __stcg(reinterpret_cast<uint4*>(c.hot_rec + slot * RB) + off, pre[u]);
                                if (off == 0) c.hot_tag[slot] = g;
                            }
                        }
                    }
                }
            }
            __syncthreads();  // batch kb_ and its meta are in shared memory
            issue(kb_ + 1);  // the next batch (nothing past the last)
            const int r0 = f0 + kb_ * kBatchRecs;
            const int nb = min(kBatchRecs, f1 - r0);
            const uint8_t* buf = s_rec + (kb_ & 1) * kFetchBatchBytes;
            const float* sbase = s_base + (kb_ & 1) * kBatchRecs * kDim;
            const uint32_t* rbits = s_rbits + (kb_ & 1) * kBatchRecs;
            // TQ-QKV: token u's sketch words and weight (0 for a slot that is no token)
            auto tok_sketch = [&](int u, uint4& wd, float& wt) {  // (gathered with the batch)
                wd = s_tsk[kb_ & 1][u];
                wt = kQjlScale * s_tnm[kb_ & 1][u];
            };
            // one recovered token: validity, RoPE'd key and rotated-frame value
            auto token = [&](int u, float kv[8], float vv[8]) -> bool {
                const int rec = u / N, n = u - rec * N;
                const int g = s_sel[r0 + rec];
                const int t = g * N + n;
                const bool ok = (g >= 0) & (t < c.T) & (((rbits[rec] >> n) & 1u) == 0u);
                const uint8_t* rp = buf + rec * RB;
                const float* norms = reinterpret_cast<const float*>(rp + N * 128);
                const uint16_t* kr = reinterpret_cast<const uint16_t*>(rp + n * 64);
                const uint16_t* vr = reinterpret_cast<const uint16_t*>(rp + N * 64 + n * 64);
                unpack4(kr[l], kr[16 + l], c4, 1.0f, kv);
                if constexpr (kRot) fwht(kv, kFull);
                const float kn = norms[n] * (kRot ? kRsqrtD : 1.f);
#pragma unroll
                for (int i = 0; i < 8; ++i) kv[i] *= sg[i] * kn;
                {   // RoPE at t = g N + n: base angle (per record) plus offset n omega
                    float4 cs = *reinterpret_cast<const float4*>(sbase + rec * kDim + 4 * l);
                    float4 sn = *reinterpret_cast<const float4*>(sbase + rec * kDim + 64 + 4 * l);
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
                return ok;
            };
            const int nt = nb * N;
            uint4 twa = make_uint4(0, 0, 0, 0), twb = twa;  // next pair's sketches (TQ-QKV)
            float tga = 0.f, tgb = 0.f;
            if constexpr (kQJL) {
                tok_sketch(min(hw, nt - 1), twa, tga);
                tok_sketch(min(hw + NH, nt - 1), twb, tgb);
            }
#pragma unroll 1
            for (int blk = 0; blk < nt; blk += 2 * NH) {
                const int ua = blk + hw, ub = ua + NH;
                float ka[8], kb[8], va[8], vb[8], xa[R], xb[R];
                const bool oka = token(min(ua, nt - 1), ka, va) && ua < nt;
                const bool okb = token(min(ub, nt - 1), kb, vb) && ub < nt;
                if constexpr (kQJL) {
                    const uint4 wa = twa, wb = twb;
                    const float ga = tga, gb = tgb;
                    if (blk + 2 * NH < nt) {
                        tok_sketch(min(ua + 2 * NH, nt - 1), twa, tga);
                        tok_sketch(min(ub + 2 * NH, nt - 1), twb, tgb);
                    }
                    float ca[8], cb[8];
                    sketch_signs(wa, ga, ca);
                    sketch_signs(wb, gb, cb);
                    pair_logits_qjl<R>(qr, ka, kb, sq, ca, cb, kLogitScaleLog2, xs, xa, xb);
                } else {
                    pair_logits<R>(qr, ka, kb, kLogitScaleLog2, xs, xa, xb);
                }
                sm.add2(xa, va, oka, xb, vb, okb);
            }
            __syncthreads();  // batch kb_ consumed: its buffer may be refilled
        }
    }

    // 6. merge the two halves of each warp, then the warps, into this split's
    //    partial of each query head, rotate it back to the original frame, and
    //    push its quads to the splits that own them
#pragma unroll
    for (int j = 0; j < R; ++j) {
        const float mo = __shfl_xor_sync(kFull, sm.m[j], 16);
        const float lo = __shfl_xor_sync(kFull, sm.l[j], 16);
        const float M = fmaxf(sm.m[j], mo);
        const float ws = merge_weight(sm.m[j], M), wo = merge_weight(mo, M);
        sm.l[j] = sm.l[j] * ws + lo * wo;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float ao = __shfl_xor_sync(kFull, sm.acc[j][i], 16);
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
    if (!kRoute) cluster_wait();  // every CTA of the cluster runs: remote stores may start
    const int P = inbox_stride(S);
    if (tid < R * 32) {  // warp j: this split's partial of query head j, 4 dims (a quad) per lane
        const int j = tid >> 5, q4 = tid & 31;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) M = fmaxf(M, s_part[((size_t)w * R + j) * hsq::kPartStride + 128]);
        float Lsum = 0.f;
        float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            const float* p = s_part + ((size_t)w * R + j) * hsq::kPartStride;
            const float wt = merge_weight(p[128], M);
            const float4 v = *reinterpret_cast<const float4*>(p + 4 * q4);
            Lsum += p[129] * wt;
            A.x += v.x * wt; A.y += v.y * wt; A.z += v.z * wt; A.w += v.w * wt;
        }
        if constexpr (kRot) {  // back to the original frame (linear, so before the merge): Pi^T = diag(s) H / sqrt(d)
            fwht_quad(A);
            const float* sq = sg + (q4 < 16 ? 0 : 4);  // this thread's signs of dims 4 q4 .. 4 q4 + 3
            A.x *= sq[0] * kRsqrtD; A.y *= sq[1] * kRsqrtD; A.z *= sq[2] * kRsqrtD; A.w *= sq[3] * kRsqrtD;
        }
        const int owner = ((q4 + 1) * S + 31) / 32 - 1;  // the split whose quads include quad q4
        float* dst = cluster.map_shared_rank(s_inbox, owner) + ((size_t)j * S + s) * P;
        *reinterpret_cast<float4*>(dst + 4 * (q4 - quad0(owner, S))) = A;
        if (q4 < S) {
            float* row = cluster.map_shared_rank(s_inbox, q4) + ((size_t)j * S + s) * P;
            row[P - 4] = M;
            row[P - 3] = Lsum;
        }
    }
    cluster.sync();  // every partial is in its owners' inboxes; no remote access follows

    // this split's quads of every query head: merge the S partials and store,
    // four threads per (head, quad), each over every fourth split, combined by
    // shuffles (loop bounds uniform: a partial past S weighs nothing)
    const int nq = quad0(s + 1, S) - quad0(s, S);
    const int nitems = R * nq;
#pragma unroll 1
    for (int base = 0; base < 4 * nitems; base += NT) {
        if (base + (tid & ~31) >= 4 * nitems) break;  // (whole warps)
        const int u = base + tid, item = u >> 2, sub = u & 3;
        const bool live = item < nitems;
        const int it = live ? item : nitems - 1;
        const int j = it / nq, kq = it - j * nq;
        const float* in = s_inbox + (size_t)j * S * P;
        float M = -INFINITY;
#pragma unroll 1
        for (int r0 = 0; r0 < S; r0 += 4) {
            const int r = min(r0 + sub, S - 1);
            M = fmaxf(M, r0 + sub < S ? in[r * P + P - 4] : -INFINITY);
        }
        M = fmaxf(M, __shfl_xor_sync(kFull, M, 1));
        M = fmaxf(M, __shfl_xor_sync(kFull, M, 2));
        float Lsum = 0.f;
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
        for (int r0 = 0; r0 < S; r0 += 4) {
            const int r = min(r0 + sub, S - 1);
            const float wt = r0 + sub < S ? merge_weight(in[r * P + P - 4], M) : 0.f;
            const float4 x = *reinterpret_cast<const float4*>(in + r * P + 4 * kq);
            Lsum += in[r * P + P - 3] * wt;
            o.x += x.x * wt; o.y += x.y * wt; o.z += x.z * wt; o.w += x.w * wt;
        }
#pragma unroll
        for (int d = 1; d < 4; d <<= 1) {
            Lsum += __shfl_xor_sync(kFull, Lsum, d);
            o.x += __shfl_xor_sync(kFull, o.x, d);
            o.y += __shfl_xor_sync(kFull, o.y, d);
            o.z += __shfl_xor_sync(kFull, o.z, d);
            o.w += __shfl_xor_sync(kFull, o.w, d);
        }
        if (live && sub == 0) {
            const float inv = Lsum > 0.f ? 1.0f / Lsum : 0.f;
            *reinterpret_cast<float4*>(a.out + ((size_t)b * c.Hq + h * R + j) * kDim + 4 * (quad0(s, S) + kq)) =
                make_float4(o.x * inv, o.y * inv, o.z * inv, o.w * inv);
        }
    }
}


// ---------------------------------------------------------------------------
// Host side: launch plan and launch.
// ---------------------------------------------------------------------------

using DecodeFn = void (*)(CacheView, DecodeArgs, Tables);

// at: room for two attributes (the cluster shape, and with overlap the
// programmatic stream serialization of hsq_config.overlap_launch).
cudaLaunchConfig_t decode_config(int S, int bh, int threads, size_t smem, cudaStream_t st, cudaLaunchAttribute* at,
                                 bool overlap = false) {
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(S, bh, 1);
    lc.blockDim = dim3(threads, 1, 1);
    lc.dynamicSmemBytes = smem;
    lc.stream = st;
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = S;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    lc.attrs = at;
    lc.numAttrs = 1;
    if (overlap) {
        at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        at[1].val.programmaticStreamSerializationAllowed = 1;
        lc.numAttrs = 2;
    }
    return lc;
}

// Best cluster size for one kernel variant: the largest S <= s_hi whose
// bh clusters are all resident at once (one wave); when none gives one wave,
// the smallest S that can launch (least per-head overhead across waves).  A
// fixed n_splits takes the largest launchable S.  0: nothing launchable.
// The kernel variant of the context's codec.
template <int R, int N, bool kRoute, bool kStaged>
DecodeFn decode_fn(bool rot, bool qjl, bool hot) {
    if constexpr (kRoute) {  // the hot-group table: TurboQuant, TQ-KV, fused step only
        if (hot) return decode_kernel<R, N, kRoute, kStaged, true, false, true>;
    }
    if (qjl) return decode_kernel<R, N, kRoute, kStaged, true, true>;  // TQ-QKV: TurboQuant only
    return rot ? decode_kernel<R, N, kRoute, kStaged, true> : decode_kernel<R, N, kRoute, kStaged, false>;
}

template <int R, int N, bool kRoute, bool kStaged>
int best_splits(hsq_ctx* ctx, int G, int T, int bh, int s_hi) {
    const void* fn = (const void*)decode_fn<R, N, kRoute, kStaged>(ctx->cfg.codec != HSQ_CODEC_PLAIN, ctx->cfg.qjl != 0,
                                                                   ctx->cfg.hot_slots > 0);
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, fn) != cudaSuccess) return 0;
    if (hsq::allow_big_clusters(fn, ctx->device) != cudaSuccess) return 0;
    const size_t cap = (size_t)ctx->smem_optin > fa.sharedSizeBytes ? ctx->smem_optin - fa.sharedSizeBytes : 0;
    const int fl = kStaged ? (kStagedFlags | (ctx->cfg.qjl ? kStageSketch : 0)) : 0;
    int last = 0;
    for (int S = s_hi; S >= 1; --S) {
        const size_t smem = decode_layout<R, N>(G, T, S, ctx->cfg.max_l1, ctx->cfg.beta, kRoute, fl).total;
        if (smem > cap) continue;
        if (hsq::raise_smem_limit(fn, ctx->device, smem) != cudaSuccess) continue;
        cudaLaunchAttribute at[2];
        cudaLaunchConfig_t lc = decode_config(S, bh, dec_threads<R>(), smem, 0, at);
        int nc = 0;
        if (cudaOccupancyMaxActiveClusters(&nc, fn, &lc) != cudaSuccess || nc < 1) continue;
        if (ctx->cfg.n_splits > 0 || nc >= bh) return S;
        last = S;
    }
    return last;
}

// Launch plan for B sequences laid out for T tokens (the capacity; cached per
// shape): staged inputs when some cluster size fits shared memory, else in place.
template <int R, int N, bool kRoute>
hsq_ctx::Plan decode_plan(hsq_ctx* ctx, int B, int T, int heads) {
    for (const auto& e : ctx->plans)
        if (e.B == B && e.T == T && e.route == (int)kRoute) return e;
    const int G = hsq::groups_of(T, N);
    const int bh = B * heads;
    const int fixed = ctx->cfg.n_splits;
    const int s_hi = std::max(1, std::min(fixed > 0 ? fixed : kMaxSplits, std::max(G, 1)));
    hsq_ctx::Plan plan{B, T, (int)kRoute, 0, 1};
    plan.S = best_splits<R, N, kRoute, true>(ctx, G, T, bh, s_hi);
    if (plan.S == 0) {
        plan.staged = 0;
        plan.S = best_splits<R, N, kRoute, false>(ctx, G, T, bh, s_hi);
    }
    cudaGetLastError();
    ctx->plans.push_back(plan);
    return plan;
}

template <int R, int N, bool kRoute, bool kStaged>
hsq_status launch_decode(hsq_ctx* ctx, const CacheView& v, const DecodeArgs& a, int S, cudaStream_t st) {
    const DecodeLayout L = decode_layout<R, N>(v.G, v.cap, S, v.max_l1, v.beta, kRoute,
                                               kStaged ? (kStagedFlags | (v.qjl_s ? kStageSketch : 0)) : 0);
    const DecodeFn kern = decode_fn<R, N, kRoute, kStaged>(v.rot != 0, v.qjl_s != nullptr, v.hot_tag != nullptr);
    const void* fn = (const void*)kern;
    cudaError_t e = hsq::raise_smem_limit(fn, ctx->device, L.total);
    if (e != cudaSuccess) return hsq::cuda_fail(ctx, e, "cudaFuncSetAttribute(decode)");
    cudaLaunchAttribute at[2];
    const cudaLaunchConfig_t lc =
        decode_config(S, v.B * v.Hkv, dec_threads<R>(), L.total, st, at, ctx->cfg.overlap_launch != 0);
    const Tables tb = make_tables(ctx);
    e = cudaLaunchKernelEx(&lc, kern, v, a, tb);
    if (e != cudaSuccess) return hsq::cuda_fail(ctx, e, "decode launch");
    return HSQ_OK;
}

template <int R, int N>
hsq_status decode_run_n(hsq_ctx* ctx, const CacheView& v, const DecodeArgs& a, bool route, cudaStream_t st,
                        bool* launched) {
    *launched = false;
    const hsq_ctx::Plan p = route ? decode_plan<R, N, true>(ctx, v.B, v.cap, v.Hkv)
                                  : decode_plan<R, N, false>(ctx, v.B, v.cap, v.Hkv);
    if (p.S == 0) return HSQ_OK;
    *launched = true;
    if (route) return p.staged ? launch_decode<R, N, true, true>(ctx, v, a, p.S, st)
                               : launch_decode<R, N, true, false>(ctx, v, a, p.S, st);
    return p.staged ? launch_decode<R, N, false, true>(ctx, v, a, p.S, st)
                    : launch_decode<R, N, false, false>(ctx, v, a, p.S, st);
}

template <int R>
hsq_status decode_run(hsq_ctx* ctx, const hsq_cache* cache, const float* q, const int32_t* pos, int32_t* sel,
                      float* out, bool route, bool from_staging, cudaStream_t st, bool* launched) {
    const CacheView v = make_sel_view(ctx, cache);
    const DecodeArgs a{q, pos, sel, out, ctx->d_err, from_staging ? 1 : 0};
    return v.N == 16 ? decode_run_n<R, 16>(ctx, v, a, route, st, launched)
                     : decode_run_n<R, 8>(ctx, v, a, route, st, launched);
}

}  // namespace

// Instantiates the decode step for head ratio R as hsq::decode_run_r<R>.
#define HSQ_DEFINE_DECODE(R)                                                                              \
    namespace hsq {                                                                                       \
    hsq_status decode_run_r##R(hsq_ctx* ctx, const hsq_cache* cache, const float* q, const int32_t* pos,  \
                               int32_t* sel, float* out, bool route, bool from_staging, cudaStream_t st,   \
                               bool* launched) {                                                          \
        return decode_run<R>(ctx, cache, q, pos, sel, out, route, from_staging, st, launched);            \
    }                                                                                                     \
    }
