/*
 * hsq.h -- C ABI of the HSQ (Hierarchical Semantic Quantization, "Tamarin")
 * compressed-KV library for GB300 (sm_103a).
 *
 * The operations follow the decode process of the Tamarin (HSQ) technical
 * summary (gist.science rs-10297225), section 2 "Method":
 *   - three-tier cache: L1 focal tier (GPU, 4-bit), L2 summary tier (GPU,
 *     3-bit, one key/value pair per group of N in {8, 16}), L3 archive of
 *     4-bit originals of every compressed token in host RAM;
 *   - decode: (1) a per-head router scores the L2 summary keys against the
 *     current query, (2) the top-beta groups' originals are fetched from L3,
 *     dequantised on the GPU and rotated to their positions, (3) attention
 *     runs over L1 tokens, L2 summaries and the recovered originals, with the
 *     summaries of fetched groups masked out.
 * Quantisation is TurboQuant as described in "Ablation, Statistical
 * Inference, and Validation for KV-Cache Compression" (gist.science
 * 2607.09683), experimental setup item 1: a randomised Walsh-Hadamard
 * rotation, then a data-oblivious Beta Lloyd-Max scalar codebook.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - head_dim d = 128.  Hq query heads, Hkv KV heads, r = Hq / Hkv; query
 *    head j reads KV head j / r.
 *  - A stored vector x is (n, codes): n = ||x|| as float32, codes = the
 *    b-bit indices of Pi (x / n), Pi = H diag(s) / sqrt(d), H the Sylvester
 *    Hadamard matrix and s the layer's +-1 sign vector.  A code is the number
 *    of codebook boundaries strictly below the coordinate.  A zero vector is
 *    n = 0 with every code 2^(b-1) - 1.
 *  - Codes are packed as a little-endian bit string: code i occupies bits
 *    [b*i, b*i + b).  A 4-bit vector takes 64 bytes, a 3-bit vector 48.
 *  - Keys enter pre-RoPE; RoPE is the rotate-half form pairing (i, i + 64)
 *    with omega_i = theta^(-2i/d).
 *  - Groups are positional blocks [gN, gN + N) over the whole context,
 *    G = ceil(T / N).  A group's members are its tokens outside L1; a group
 *    without members is empty and is never routed.
 *  - Every pointer in hsq_cache and every array argument is caller-owned.
 *    The library owns only the context (codebooks, RoPE tables, scratch).
 *  - Every call is asynchronous on the given stream and returns a status;
 *    none aborts, asserts or traps.  Argument errors are reported before
 *    anything is enqueued.  Device-side checks (bad selection indices, a
 *    position outside the RoPE tables, an L1 set over capacity) set a
 *    context error word that hsq_sync_status() reports.
 *  - One context serves one stream at a time: its scratch is shared by the
 *    calls made with it.
 */
#ifndef HSQ_H
#define HSQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t / cudaEvent_t compatible handles (NULL = legacy default stream). */
typedef struct CUstream_st* hsq_stream_t;

typedef enum {
    HSQ_OK = 0,
    HSQ_ERR_INVALID = 1,      /* bad argument or configuration */
    HSQ_ERR_CUDA = 2,         /* a CUDA runtime call failed (see hsq_last_error) */
    HSQ_ERR_NOMEM = 3,        /* device allocation failed at hsq_create */
    HSQ_ERR_TIMEOUT = 4,      /* reserved: a bounded device wait ran out */
    HSQ_ERR_DEVICE_CHECK = 5, /* a device-side check failed (see hsq_sync_status) */
    HSQ_ERR_UNSUPPORTED = 6   /* valid but not built (e.g. an r outside {1,2,4,5,8}) */
} hsq_status;

typedef enum { HSQ_DTYPE_F32 = 0, HSQ_DTYPE_BF16 = 1 } hsq_dtype;

enum { HSQ_HEAD_DIM = 128, HSQ_MAX_BETA = 512, HSQ_MAX_SPLITS = 16 };

typedef enum { HSQ_CODEC_TQ = 0, HSQ_CODEC_PLAIN = 1 } hsq_codec;

/* Bits of the device error word (hsq_sync_status fills *device_word). */
enum {
    HSQ_DEVERR_SEL = 1,       /* selection entry out of range or not ascending: treated as -1 */
    HSQ_DEVERR_POS = 2,       /* position outside [0, max_pos): clamped */
    HSQ_DEVERR_L1_OVER = 4,   /* more L1 tokens than max_l1: extra tokens dropped from L1 */
    HSQ_DEVERR_WAIT = 8,      /* a bounded wait of the prefill attention kernel (on its bulk
                                 copies or its tensor-core work) ran out: its output is not
                                 written */
    HSQ_DEVERR_GROW = 16      /* hsq_append: the token leaving the recent window was not in L1
                                 (the cache was not encoded with that window): L1 left as is */
};

/* Flags of hsq_decode_attn. */
enum {
    HSQ_ATTN_FROM_STAGING = 1 /* read fetched records from cache->staging (filled by
                                 hsq_fetch_dequant) instead of gathering them from L3 */
};

/* Host-only fault injection (hsq_debug_set_fault). */
enum {
    HSQ_FAULT_ALLOC = 1,      /* hsq_create fails with HSQ_ERR_NOMEM before any CUDA call */
    HSQ_FAULT_FETCH = 2       /* hsq_fetch_dequant / hsq_decode_attn return HSQ_ERR_CUDA
                                 without launching */
};

typedef struct hsq_config {
    int n_q_heads;      /* Hq >= 1 */
    int n_kv_heads;     /* Hkv >= 1, Hq % Hkv == 0, r = Hq / Hkv in {1, 2, 4, 5, 8} */
    int head_dim;       /* must be 128 */
    int group_n;        /* N: 8 or 16 (group size of the L2 tier) */
    int beta;           /* groups fetched per KV head per step, 1..HSQ_MAX_BETA */
    int bits_l1l3;      /* must be 4 (L1 and L3 precision) */
    int bits_l2;        /* must be 3 (L2 summary precision) */
    double rope_theta;  /* RoPE base, > 0 */
    int max_batch;      /* largest B any cache of this context has */
    int max_ctx;        /* largest T */
    int max_l1;         /* L1 slots per sequence */
    int max_pos;        /* exclusive bound on positions (context + decode steps), <= 2^24 */
    int n_splits;       /* decode splits (CTAs of one thread-block cluster) per (b, KV head):
                           0 = automatic, else an upper bound in [1, HSQ_MAX_SPLITS] */
    /* Decode-time growth (hsq_append).  The L1 set then is: positions below
       l1_sinks, the positions marked at encode time, and the recent window
       [T - l1_recent, T), which slides by one with every appended token. */
    int l1_sinks;       /* >= 0 */
    int l1_recent;      /* >= 0; 0 = caches of this context do not grow */
    /* How a KV head's routing score combines its query heads: 0 = their sum
       (one dot with the summed rotated queries), 1 = their maximum (a group
       counts as much as it does for its best query head). */
    int route_max;
    /* Codec of every tier (hsq_codec).  HSQ_CODEC_TQ: TurboQuant, the unit
       vector rotated by Pi = H diag(s) / sqrt(128) before the codebook
       ("Tamarin (HSQ)", key components; "Ablation, Statistical Inference, and
       Validation for KV-Cache Compression", experimental setup, item 1).
       HSQ_CODEC_PLAIN: Plain-KV, the same codebook on the unrotated unit
       vector (the second page's scalar quantisation without rotation); the
       signs buffer is then not read. */
    int codec;
    /* 1: per-query-head routing -- every query head selects its own beta
       groups by its own score against its KV head's summaries and attends
       with that selection (the router of "Tamarin (HSQ)", decode process,
       step 1, is per head).  sel, scores and staging then have one row per
       query head ([B][Hq][...]) instead of one per KV head, and each query
       head fetches its own records.  0: one selection per KV head.  Not
       together with route_max. */
    int route_per_head;
    /* 1: TQ-QKV ("Ablation, Statistical Inference, and Validation for
       KV-Cache Compression", key contributions, item 1) -- every 4-bit key
       (L1 and L3) also keeps a 1-bit Johnson-Lindenstrauss sketch of its
       quantisation residual rho, taken in the frame its logit is computed in
       and rotated by the codec (L3: Pi RoPE(k_t - k^_t, t); L1: Pi (RoPE(k_t, t)
       - k^)): 128 bits (S rho >= 0) and |rho|, S = cache->qjl_s.  A token's
       logit then adds sqrt(pi/2) / 128 * |rho| * sum_i (S Pi q^r)_i sign_i
       before the 1/sqrt(128) scale (an unbiased estimate of q^r . residual).
       Needs codec HSQ_CODEC_TQ.  hsq_encode writes the sketches (the key
       input is read a second time); hsq_append refuses it (HSQ_ERR_UNSUPPORTED).
       0: TQ-KV. */
    int qjl;
    /* Hot-group table of the fused decode step (hsq_decode_step only): 0 = none;
       else a power of two in [16, 1024], the slots of a direct-mapped device
       copy of recently fetched L3 records per (sequence, KV head).  Group g
       lives in slot g mod hot_slots.  A step reads a selected group's record
       from its slot when the slot's tag is g (no host-link transfer); a record
       it fetched from L3 is copied into its slot, and the tag set, when no
       other group of the step's selection maps to that slot (so a step never
       reads and writes one slot).  Results are bit-identical with and without
       the table.  The cache then needs hot_rec and hot_tag; hsq_encode empties
       the table, hsq_append drops the group it writes.  An engineering
       addition (the pages describe no such cache): it saves host-link bytes
       when consecutive steps select overlapping groups.  Needs codec
       HSQ_CODEC_TQ, qjl 0 and route_per_head 0. */
    int hot_slots;
    /* 1: launch the decode kernels (hsq_decode_step, hsq_decode_attn) with
       programmatic stream serialization.  Such a launch may be scheduled onto
       the GPU while the stream's preceding kernel still runs; the kernel then
       waits, before its first read or write of global memory, until that
       kernel has completed and its writes are visible, so results are the
       same as with 0.  Once all of its own CTAs are running it lets the
       stream's next kernel be scheduled the same way (that kernel, when it is
       another library's, must wait on its own).  It hides the launch gap
       between decode steps issued back to back (one per layer), directly or
       captured in a CUDA graph.  0: ordinary stream order. */
    int overlap_launch;
} hsq_config;

/*
 * Cache buffers of one layer.  Sizes in bytes come from hsq_cache_sizes(),
 * in the order of enum hsq_buffer.  All device buffers are plain device
 * memory; l3 is either device memory or page-locked host memory mapped into
 * the device address space (cudaHostAlloc / torch pin_memory), read by the
 * GPU in place (zero copy); l3 must be 16-byte aligned (HSQ_ERR_INVALID
 * otherwise: records are read in 16-byte chunks).
 */
typedef struct hsq_cache {
    int B;                    /* sequences in this cache, 1..max_batch */
    int T;                    /* tokens per sequence, positions 0..T-1, 1..max_ctx */
    /* L1 focal tier */
    uint8_t* l1_kc;           /* [B][Hkv][max_l1][64]  4-bit codes of RoPE(k_t, t) */
    uint8_t* l1_vc;           /* [B][Hkv][max_l1][64]  4-bit codes of v_t */
    float* l1_kn;             /* [B][Hkv][max_l1]      key norms */
    float* l1_vn;             /* [B][Hkv][max_l1]      value norms */
    int32_t* l1_pos;          /* [B][max_l1]           L1 positions (ascending after encode) */
    int32_t* l1_count;        /* [B]                   L1 size per sequence */
    /* L2 summary tier */
    uint8_t* l2_kc;           /* [B][Hkv][G][48]  3-bit codes of the members' mean RoPE'd key */
    uint8_t* l2_vc;           /* [B][Hkv][G][48]  3-bit codes of the members' mean value */
    float* l2_kn;             /* [B][Hkv][G] */
    float* l2_vn;             /* [B][Hkv][G] */
    uint8_t* l2_cnt;          /* [B][G] members per group (0 = empty) */
    /* L3 archive: group-major records, one per (b, h, g), of N*136 bytes:
       K codes [N][64] | V codes [N][64] | K norms [N] f32 | V norms [N] f32.
       Slots past T hold the zero-vector encoding. */
    uint8_t* l3;
    int l3_on_host;           /* 1 = page-locked host memory, 0 = device memory */
    /* L1 membership: bit (t & 31) of word [b][t >> 5]; bits at t >= T are ignored */
    uint32_t* l1_bitmap;      /* [B][ceil(t_cap/32)] device (hsq_append updates it) */
    const int8_t* signs;      /* [128] device, +-1: the layer's Walsh-Hadamard sign vector */
    uint8_t* staging;         /* [B][Hkv or Hq (route_per_head)][beta][N*136] device, or NULL (only needed for the
                                 staged fetch path) */
    /* Capacity and decode-time growth state (hsq_append). */
    int t_cap;                /* tokens the buffers are laid out for, T <= t_cap <= max_ctx
                                 (0 = T): every G above is ceil(t_cap / N) and the bitmap has
                                 ceil(t_cap / 32) words per sequence; groups past T are empty */
    float* win_kv;            /* [B][Hkv][l1_recent][2][128] device, or NULL: the input (pre-RoPE)
                                 key and the value of each recent-window token, slot p mod
                                 l1_recent; written by hsq_encode, read and written by hsq_append */
    float* gsum;              /* [B][Hkv][260] device, or NULL: for the group holding position
                                 T - l1_recent, the float sums, in position order, of its members
                                 below that position: RoPE'd keys [128] | values [128] | member
                                 count | the window's first position at encode | pad [2] */
    /* Key-residual sketches (cfg.qjl = 1; else ignored).  Sketch words: bit i of
       the 128-bit sketch is bit (i mod 32) of word i / 32. */
    const float* qjl_s;       /* [128][128] device, row i = sketch direction i (i.i.d. N(0,1)) */
    uint32_t* l1_qs;          /* [B][Hkv][max_l1][4] device: sketches of the L1 keys' residuals */
    float* l1_qn;             /* [B][Hkv][max_l1] device: their norms */
    uint32_t* l3_qs;          /* [B][Hkv][G*N][4] device: sketches of every token's key residual */
    float* l3_qn;             /* [B][Hkv][G*N] device: their norms */
    /* Hot-group table (cfg.hot_slots > 0; else ignored). */
    uint8_t* hot_rec;         /* [B][Hkv][hot_slots][N*136] device: copies of L3 records */
    int32_t* hot_tag;         /* [B][Hkv][hot_slots] device: the group in each slot, -1 = empty */
} hsq_cache;

typedef enum {
    HSQ_BUF_L1_KC = 0, HSQ_BUF_L1_VC, HSQ_BUF_L1_KN, HSQ_BUF_L1_VN, HSQ_BUF_L1_POS,
    HSQ_BUF_L1_COUNT, HSQ_BUF_L2_KC, HSQ_BUF_L2_VC, HSQ_BUF_L2_KN, HSQ_BUF_L2_VN,
    HSQ_BUF_L2_CNT, HSQ_BUF_L3, HSQ_BUF_L1_BITMAP, HSQ_BUF_STAGING, HSQ_BUF_WIN_KV,
    HSQ_BUF_GSUM, HSQ_BUF_L1_QS, HSQ_BUF_L1_QN, HSQ_BUF_L3_QS, HSQ_BUF_L3_QN,
    HSQ_BUF_HOT_REC, HSQ_BUF_HOT_TAG, HSQ_NBUF
} hsq_buffer;

typedef struct hsq_ctx hsq_ctx;   /* opaque, library-owned */

/*
 * hsq_codebook -- the TurboQuant Beta Lloyd-Max codebook (host only, float64).
 *   Lloyd-Max for the law of one coordinate of a uniform unit vector in R^dim
 *   (Y^2 ~ Beta(1/2, (dim-1)/2)), iterated to convergence; symmetric, so the
 *   middle boundary is 0.  ("Ablation, Statistical Inference, and Validation
 *   for KV-Cache Compression", experimental setup item 1.)
 *   centroids: [2^bits] ascending; boundaries: [2^bits - 1], midpoints.
 *   bits in 1..8, dim >= 4.  Needs no GPU.  Errors: HSQ_ERR_INVALID.
 */
hsq_status hsq_codebook(int bits, int dim, double* centroids, double* boundaries);

/*
 * hsq_cache_sizes -- bytes of each buffer of a cache with B sequences of T
 *   tokens under cfg, indexed by enum hsq_buffer (for a cache that grows, T
 *   is its capacity t_cap; the growth buffers are 0 bytes when l1_recent is
 *   0).  Needs no GPU.
 *   Errors: HSQ_ERR_INVALID (bad cfg, B or T).
 */
hsq_status hsq_cache_sizes(const hsq_config* cfg, int B, int T, size_t bytes[HSQ_NBUF]);

/*
 * hsq_create -- validate cfg, build both codebooks (float64, rounded to
 *   float32 for the device) and the RoPE angle tables (float64 angles,
 *   float32 cos/sin of 256*a*omega and c*omega, combined on the device by
 *   angle addition), allocate scratch on the current device (with cfg.qjl
 *   also 64 KB for S Pi and max_batch * n_kv_heads * ceil(max_ctx / group_n)
 *   * group_n * 68 bytes for a copy of the last encode's L3 key codes and
 *   norms, read by the sketch pass).
 *   *out receives the context.  Errors: HSQ_ERR_INVALID, HSQ_ERR_NOMEM,
 *   HSQ_ERR_CUDA, HSQ_ERR_UNSUPPORTED.
 */
hsq_status hsq_create(const hsq_config* cfg, hsq_ctx** out);

/* hsq_destroy -- free the context (synchronises its device work). NULL is a no-op. */
hsq_status hsq_destroy(hsq_ctx* ctx);

/*
 * hsq_encode -- build the three tiers of one layer from pre-RoPE K and V
 *   (Tamarin summary, section 2, three-tier architecture; TurboQuant encode).
 *   K, V: device [B][Hkv][T][128] of dtype (bf16 or f32), positions 0..T-1.
 *   Reads cache->l1_bitmap and cache->signs; writes every L1, L2 and L3
 *   buffer:
 *     L3 record slot t: TQ4(k_t) and TQ4(v_t) for every token;
 *     L1 slot i (ascending position order): TQ4(RoPE(k_t, t)), TQ4(v_t);
 *     L2 group g: TQ3(mean of RoPE(k_t, t)), TQ3(mean of v_t) over members,
 *       count in l2_cnt; an empty group stores the zero vector.
 *   If l3_on_host, the records are written through the host link.  With
 *   cfg.l1_recent > 0 and win_kv / gsum set, it also stores the growth state
 *   that hsq_append continues from (the recent window's inputs and the
 *   running sums of the group at the window's trailing edge).  Groups and
 *   records past T (up to t_cap) are written empty.  With cfg.qjl it also
 *   writes the key-residual sketches (l1_qs / l1_qn, l3_qs / l3_qn) from
 *   cache->qjl_s, reading K a second time.  Under HSQ_CODEC_PLAIN every "Pi"
 *   here is the identity and signs is not read.  With cfg.hot_slots it empties
 *   the hot-group table (every hot_tag -1).
 *   Errors: HSQ_ERR_INVALID (null pointer, B/T out of range, L3 location not
 *   matching l3_on_host), HSQ_ERR_CUDA.  An L1 set larger than max_l1 sets
 *   HSQ_DEVERR_L1_OVER.
 */
hsq_status hsq_encode(hsq_ctx* ctx, const hsq_cache* cache, const void* K, const void* V,
                      hsq_dtype dtype, hsq_stream_t stream);

/*
 * hsq_append -- decode-time growth: append one token per sequence at
 *   position T (cache->T, the same for all B sequences), then T += 1 in
 *   *cache.  The pages build the three tiers from a context and leave their
 *   growth open; this call keeps the cache equal to what hsq_encode would
 *   build from the longer context with the L1 set of hsq_config (sinks,
 *   marked positions, and the recent window [T + 1 - l1_recent, T + 1)):
 *     L3 record slot T: TQ4(k) and TQ4(v);
 *     L1: TQ4(RoPE(k, T)) and TQ4(v) in the slot of the token p = T - l1_recent
 *       that leaves the window (a new slot when p < max(l1_sinks, 0));
 *     p joins group p / N: its summary is re-quantised from the members'
 *       running float sums (position order, as hsq_encode sums them);
 *     the L1 bitmap, positions and counts and l2_cnt follow;
 *     with cfg.hot_slots, the hot-group table drops group T / N of every
 *       (b, h) if it holds it (its record changed).
 *   k, v: device [B][Hkv][128] of dtype, pre-RoPE.  Needs cfg.l1_recent > 0,
 *   cache->win_kv and cache->gsum (filled by hsq_encode under this cfg),
 *   T < t_cap and T < max_pos.  L1 slots are then no longer in position
 *   order (l1_pos holds each slot's position).  Errors: HSQ_ERR_INVALID,
 *   HSQ_ERR_UNSUPPORTED (cfg.qjl), HSQ_ERR_CUDA; device checks
 *   HSQ_DEVERR_GROW, HSQ_DEVERR_L1_OVER.
 */
hsq_status hsq_append(hsq_ctx* ctx, hsq_cache* cache, const void* k, const void* v, hsq_dtype dtype,
                      hsq_stream_t stream);

/*
 * hsq_route -- per-head routing and top-beta group selection (decode
 *   process, steps 1-2).  For each (b, KV head h):
 *     s_g = sum over the head's query heads j of RoPE(q_j, pos_b) . k_hat_g
 *   (k_hat_g the dequantised summary key), computed in the rotated frame as
 *   n_g * (sum_j Pi RoPE(q_j, pos_b)) . c3[codes_g]; with cfg.route_max the
 *   maximum over j of n_g * (Pi RoPE(q_j, pos_b)) . c3[codes_g] instead
 *   (hsq_decode_step then runs hsq_route and hsq_decode_attn; the no-alloc
 *   routing call refuses it); empty groups score -inf.  With
 *   cfg.route_per_head every query head j has its own row:
 *   s_g = n_g * (Pi RoPE(q_j, pos_b)) . c3[codes_g] of its KV head, and sel,
 *   scores_opt (and, in the calls below, staging and the fetched outputs)
 *   have Hq rows in place of Hkv.
 *   sel[b][h][0..beta) = the beta largest scores, ties to the lower group,
 *   listed in ascending group order, -1 padded when fewer are non-empty.
 *   q: [B][Hq][128] f32; pos: [B] int32 (query positions); sel:
 *   [B][Hkv][beta] int32 -- each device memory or page-locked host memory
 *   mapped at the same address (read / written in place over the host link);
 *   scores_opt: device [B][Hkv][G] f32 or NULL.  Errors: HSQ_ERR_INVALID
 *   (also for a pageable host pointer), HSQ_ERR_CUDA.
 */
hsq_status hsq_route(hsq_ctx* ctx, const hsq_cache* cache, const float* q, const int32_t* pos,
                     int32_t* sel, float* scores_opt, hsq_stream_t stream);

/*
 * hsq_fetch_dequant -- fetch the selected groups' L3 records and recover the
 *   originals (decode process, step 2).  Copies record (b, h, sel[b][h][i])
 *   to cache->staging[b][h][i] when staging is not NULL, and optionally
 *   writes, for token t = g*N + n:
 *     k_out_opt [B][Hkv][beta][N][128] f32: RoPE(Pi^T n c4[codes], t), original frame;
 *     v_out_opt [same] f32: Pi^T n c4[codes], original frame;
 *     valid_opt [B][Hkv][beta][N] u8: 1 unless sel = -1, t >= T or t in L1.
 *   Slots with sel = -1 or t >= T are written as zeros.  All outputs device.
 *   Errors: HSQ_ERR_INVALID, HSQ_ERR_CUDA.
 */
hsq_status hsq_fetch_dequant(hsq_ctx* ctx, const hsq_cache* cache, const int32_t* sel,
                             float* k_out_opt, float* v_out_opt, uint8_t* valid_opt,
                             hsq_stream_t stream);

/*
 * hsq_recover -- recover the originals of groups [g0, g0 + ng) from L3
 *   ("Tamarin (HSQ) - reversible hierarchical KV-cache compression": the
 *   archive keeps every compressed token recoverable).  For token
 *   t = g*N + n, slot i = g - g0:
 *     k_out_opt [B][Hkv][ng][N][128] f32: Pi^T n c4[codes] of the key, pre-RoPE;
 *     v_out_opt [same] f32: the same for the value;
 *   both in the original frame; tokens t >= T are written as zeros.  L1
 *   tokens are recovered too (L3 holds every token).  Outputs: device
 *   memory or mapped page-locked host memory, at least one not NULL.
 *   Errors: HSQ_ERR_INVALID (g0 < 0, ng < 1, g0 + ng > ceil(T / N), no
 *   output), HSQ_ERR_CUDA.
 */
hsq_status hsq_recover(hsq_ctx* ctx, const hsq_cache* cache, int g0, int ng, float* k_out_opt,
                       float* v_out_opt, hsq_stream_t stream);

/*
 * hsq_decode_attn -- union attention of one decode step (decode process,
 *   step 3).  For each query head j of KV head h, one softmax with scale
 *   1/sqrt(128) over
 *     L1 tokens (key RoPE'd at encode),
 *     non-empty groups not in sel (one entry each: summary key and value),
 *     tokens t of the groups in sel that are not in L1 (key RoPE(k_t, t)
 *     recovered from L3, value v_t),
 *   split over the entries (flash-decoding) and merged by log-sum-exp.
 *   With cfg.qjl the L1 and fetched-token logits carry the sketch term
 *   (hsq_config.qjl); with cfg.route_per_head query head j attends with its
 *   own row sel[b][j] (L1, the summaries of groups not in it, the tokens of
 *   the groups in it).
 *   out: [B][Hq][128] f32 in the original frame, device memory or mapped
 *   page-locked host memory (written in place).  q, pos, sel as in
 *   hsq_route.  By default the kernel gathers the selected L3 records itself
 *   (zero-copy when L3 is on the host); with HSQ_ATTN_FROM_STAGING it reads
 *   cache->staging, which a prior hsq_fetch_dequant filled (order the two
 *   with the caller's events when they run on different streams).
 *   Errors: HSQ_ERR_INVALID, HSQ_ERR_CUDA; bad sel entries set HSQ_DEVERR_SEL.
 */
hsq_status hsq_decode_attn(hsq_ctx* ctx, const hsq_cache* cache, const float* q,
                           const int32_t* pos, const int32_t* sel, float* out, int flags,
                           hsq_stream_t stream);

/*
 * hsq_decode_step -- one whole decode step of one layer: routing, top-beta
 *   selection, gather of the selected L3 records and the union attention.
 *   sel is written exactly as hsq_route writes it (same scores, same
 *   selection) and out as hsq_decode_attn computes it.  One kernel: the S
 *   splits of a (b, h) form one thread-block cluster and select the top
 *   beta together through distributed shared memory, so no CTA waits on a
 *   CTA outside its cluster and the grid need not be co-resident.  It runs
 *   hsq_route then hsq_decode_attn under cfg.route_max, and when no
 *   cluster shape can be launched.  Per-query-head routing and TQ-QKV stay
 *   one launch.  q, pos, sel, out: as for those calls (device memory,
 *   or mapped page-locked host memory for a step with no separate copies).
 *   With cfg.hot_slots the fused launch reads and fills the cache's hot-group
 *   table (hsq_config.hot_slots); the separate calls do not use it.
 *   Errors as the two calls, and HSQ_ERR_INVALID when cfg.hot_slots is set and
 *   hot_rec or hot_tag is NULL.
 */
hsq_status hsq_decode_step(hsq_ctx* ctx, const hsq_cache* cache, const float* q,
                           const int32_t* pos, int32_t* sel, float* out, hsq_stream_t stream);

/*
 * hsq_sync_status -- synchronise `stream`, read and clear the device error
 *   word.  Returns HSQ_ERR_DEVICE_CHECK if any bit was set (the bits go to
 *   *device_word when it is not NULL), HSQ_ERR_CUDA on a CUDA error.
 */
hsq_status hsq_sync_status(hsq_ctx* ctx, hsq_stream_t stream, int* device_word);

/*
 * hsq_prefill -- a prompt's prefill with HSQ: the dense causal attention of
 *   the prompt and, when cache is not NULL, the encode of its K/V into the
 *   cache ("Tamarin (HSQ)" technical summary, section 4, results: the prefill
 *   overhead of compressing the prompt).  The attention is the model's
 *   ordinary one: out[b, j, t] = sum over s <= t of
 *   softmax_s(RoPE(q_{j,t}, t) . RoPE(k_{h,s}, s) / sqrt(128)) v_{h,s},
 *   h = j / (Hq / Hkv), computed on the tensor cores with fp32-level
 *   accuracy (queries, keys and probabilities split into two bf16 terms).
 *   With a cache, the encode is hsq_encode's (the same codes) and the same
 *   pass over K/V writes the attention's key and value operands, so K/V are
 *   read once.  With cache NULL only the attention runs.
 *   Q: [B, Hq, T, 128] bf16 pre-RoPE queries at positions 0..T-1; K, V:
 *   [B, Hkv, T, 128] bf16 pre-RoPE keys and values (device memory); out:
 *   [B, Hq, T, 128] float32 (device).  workspace: device memory of at least
 *   hsq_prefill_workspace_size bytes, 256-byte aligned, caller-owned, holding
 *   the operand images between the calls' kernels (its contents are not
 *   needed afterwards).  B <= max_batch, T <= max_pos; with a cache, B and T
 *   equal the cache's.  Asynchronous on `stream`.  Errors: HSQ_ERR_INVALID
 *   (NULL pointers, sizes, alignment, a small workspace, L3 placement as for
 *   hsq_encode), HSQ_ERR_CUDA.  A bounded wait inside the attention kernel
 *   that runs out sets HSQ_DEVERR_WAIT (hsq_sync_status).
 */
hsq_status hsq_prefill_workspace_size(const hsq_ctx* ctx, int B, int T, size_t* bytes);
hsq_status hsq_prefill(hsq_ctx* ctx, const hsq_cache* cache, const void* Q, const void* K, const void* V, int B,
                       int T, float* out, void* workspace, size_t workspace_bytes, hsq_stream_t stream);

/*
 * hsq_route_noalloc -- hsq_route for callers that cannot allocate device memory.
 *   The pages have no counterpart: this is an interface of this library only.
 *   Who needs it: a caller that owns all device memory through its own pool
 *   and fails any later cudaMalloc, or one that must not let a library call
 *   synchronise the device (cudaMalloc may).  It takes no context and calls
 *   no cudaMalloc, cudaFree or other allocating routine.
 *   Same inputs and output as hsq_route (cfg describes the cache; scores are
 *   not returned).  The query's RoPE angles are evaluated in float64 inside
 *   the kernel, so scores agree with hsq_route to fp32 rounding and sel is
 *   identical except for near-ties of the beta-th score.  A position outside
 *   [0, cfg->max_pos) is clamped into it, as hsq_route clamps it, but is not
 *   reported (there is no device error word without a context).
 *   Scratch: a fixed array of HSQ_NOALLOC_SCRATCH_BYTES in device memory,
 *   defined in the library and held by every GPU that loads it until the
 *   process exits.  It holds 256-byte-rounded B*Hkv tickets plus the
 *   B*Hkv*ceil(T/N) float32 scores; larger caches are rejected with
 *   HSQ_ERR_INVALID before anything is enqueued.  Every call shares that
 *   array: calls whose kernels overlap on the GPU (other streams, other
 *   threads) race and must be ordered by the caller.  The tickets are
 *   cleared (cudaMemsetAsync on `stream`) at the start of each call.
 *   The first call on a device sets that device up (looks up the array's
 *   device address, synchronously; the codebook is passed to the kernel by
 *   value); make that first call outside any stream capture.  The set-up is
 *   repeated when the device's CUDA context has changed since (after a
 *   device reset), so the same rule holds for the first call after a reset.
 *   Errors: HSQ_ERR_INVALID,
 *   HSQ_ERR_UNSUPPORTED, HSQ_ERR_CUDA (text via hsq_last_error(NULL)).
 */
enum { HSQ_NOALLOC_SCRATCH_BYTES = 4 << 20 };
hsq_status hsq_route_noalloc(const hsq_config* cfg, const hsq_cache* cache, const float* q,
                             const int32_t* pos, int32_t* sel, hsq_stream_t stream);

/* hsq_last_error -- text of the last error of ctx (or of the process when ctx is NULL). */
const char* hsq_last_error(const hsq_ctx* ctx);

/* hsq_debug_set_fault -- process-wide host-side fault injection mask (HSQ_FAULT_*). */
hsq_status hsq_debug_set_fault(unsigned mask);

/* hsq_version -- library version string. */
const char* hsq_version(void);

#ifdef __cplusplus
}
#endif

#endif /* HSQ_H */
