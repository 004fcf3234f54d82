// Host-only parts of the HSQ library: the TurboQuant codebook, RoPE tables,
// buffer sizes and argument validation.  Nothing here touches a GPU, so all
// of it is callable (and tested) on a machine without one.
//
// Codebook: "Ablation, Statistical Inference, and Validation for KV-Cache
// Compression" (technical summary, experimental setup item 1) quantises each
// coordinate of the Walsh-Hadamard-rotated unit vector with a data-oblivious
// Beta Lloyd-Max codebook.  The law of one coordinate Y of a uniform unit
// vector in R^d has density f(y) = C_d (1 - y^2)^((d-3)/2) on [-1, 1],
// C_d = Gamma(d/2) / (sqrt(pi) Gamma((d-1)/2)).  Cell probabilities are
// integrated here with composite Gauss-Legendre quadrature; the first moment
// of a cell has the closed form C_d / (d-1) * ((1-a^2)^((d-1)/2) - (1-b^2)^((d-1)/2)).

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "hsq_internal.h"

namespace hsq {

namespace {

// Gauss-Legendre nodes and weights on [-1, 1] by Newton's method on P_n.
void gauss_legendre(int n, std::vector<double>& x, std::vector<double>& w) {
    x.assign(n, 0.0);
    w.assign(n, 0.0);
    const double pi = 3.14159265358979323846;
    for (int i = 0; i < (n + 1) / 2; ++i) {
        double z = std::cos(pi * (i + 0.75) / (n + 0.5));
        double dp = 0.0;
        for (int it = 0; it < 100; ++it) {
            double p0 = 1.0, p1 = 0.0;
            for (int k = 1; k <= n; ++k) {  // recurrence k P_k = (2k-1) z P_{k-1} - (k-1) P_{k-2}
                double p2 = p1;
                p1 = p0;
                p0 = ((2.0 * k - 1.0) * z * p1 - (k - 1.0) * p2) / k;
            }
            dp = n * (z * p0 - p1) / (z * z - 1.0);
            double dz = p0 / dp;
            z -= dz;
            if (std::fabs(dz) < 1e-16) break;
        }
        x[i] = -z;
        x[n - 1 - i] = z;
        w[i] = w[n - 1 - i] = 2.0 / ((1.0 - z * z) * dp * dp);
    }
}

struct CoordinateLaw {
    int d;
    double C;
    std::vector<double> gx, gw;
    explicit CoordinateLaw(int dim) : d(dim) {
        C = std::exp(std::lgamma(0.5 * d) - 0.5 * std::log(3.14159265358979323846) -
                     std::lgamma(0.5 * (d - 1)));
        gauss_legendre(20, gx, gw);
    }
    double pdf(double y) const {
        double u = 1.0 - y * y;
        return u <= 0.0 ? 0.0 : C * std::pow(u, 0.5 * (d - 3));
    }
    // P(lo < Y <= hi), panels no wider than 1/256
    double mass(double lo, double hi) const {
        int panels = std::max(1, (int)std::ceil((hi - lo) * 256.0));
        double h = (hi - lo) / panels, s = 0.0;
        for (int p = 0; p < panels; ++p) {
            double a = lo + p * h, mid = a + 0.5 * h, half = 0.5 * h, acc = 0.0;
            for (size_t k = 0; k < gx.size(); ++k) acc += gw[k] * pdf(mid + half * gx[k]);
            s += acc * half;
        }
        return s;
    }
    double moment(double lo, double hi) const {
        double e = 0.5 * (d - 1);
        return C / (d - 1) * (std::pow(1.0 - lo * lo, e) - std::pow(1.0 - hi * hi, e));
    }
};

// inverse of the standard normal CDF by Newton steps on erfc
double normal_quantile(double p) {
    double x = 0.0;
    for (int it = 0; it < 60; ++it) {
        double cdf = 0.5 * std::erfc(-x / std::sqrt(2.0));
        double pdf = std::exp(-0.5 * x * x) / std::sqrt(2.0 * 3.14159265358979323846);
        double dx = (cdf - p) / pdf;
        x -= dx;
        if (std::fabs(dx) < 1e-15) break;
    }
    return x;
}

std::atomic<unsigned> g_fault{0};
std::mutex g_err_mu;
std::string g_err;

}  // namespace

bool lloyd_max(int bits, int dim, double* centroids, double* boundaries) {
    if (bits < 1 || bits > 8 || dim < 4) return false;
    const int L = 1 << bits, half = L / 2;
    CoordinateLaw law(dim);
    std::vector<double> p(half), edges(half + 1), nxt(half);
    for (int i = 0; i < half; ++i)
        p[i] = normal_quantile((half + i + 0.5) / L) / std::sqrt((double)dim);
    for (int it = 0; it < 200000; ++it) {
        edges[0] = 0.0;
        for (int i = 1; i < half; ++i) edges[i] = 0.5 * (p[i - 1] + p[i]);
        edges[half] = 1.0;
        double delta = 0.0;
        for (int i = 0; i < half; ++i) {
            nxt[i] = law.moment(edges[i], edges[i + 1]) / law.mass(edges[i], edges[i + 1]);
            delta = std::max(delta, std::fabs(nxt[i] - p[i]));
        }
        p = nxt;
        if (delta < 1e-15) break;
    }
    for (int i = 0; i < half; ++i) {
        centroids[half + i] = p[i];
        centroids[half - 1 - i] = -p[i];
    }
    for (int k = 0; k < L - 1; ++k) boundaries[k] = 0.5 * (centroids[k] + centroids[k + 1]);
    boundaries[half - 1] = 0.0;
    return true;
}

void device_codebook(float out[kCodebookFloats]) {
    double c4[16], t4[15], c3[8], t3[7];
    lloyd_max(4, kDim, c4, t4);
    lloyd_max(3, kDim, c3, t3);
    std::memset(out, 0, sizeof(float) * kCodebookFloats);
    for (int i = 0; i < 16; ++i) out[i] = (float)c4[i];
    for (int i = 0; i < 15; ++i) out[16 + i] = (float)t4[i];
    for (int i = 0; i < 8; ++i) out[32 + i] = (float)c3[i];
    for (int i = 0; i < 7; ++i) out[40 + i] = (float)t3[i];
}

void rope_tables(double theta, int max_pos, std::vector<float>& hi, std::vector<float>& lo) {
    const int half = kDim / 2;
    const int n_hi = (max_pos + kRopeLoRows - 1) / kRopeLoRows;
    hi.assign((size_t)n_hi * kRopeRowFloats, 0.f);
    lo.assign((size_t)kRopeLoRows * kRopeRowFloats, 0.f);
    for (int i = 0; i < half; ++i) {
        double w = std::pow(theta, -2.0 * i / kDim);
        for (int a = 0; a < n_hi; ++a) {
            double ang = (double)a * kRopeLoRows * w;
            hi[(size_t)a * kRopeRowFloats + i] = (float)std::cos(ang);
            hi[(size_t)a * kRopeRowFloats + half + i] = (float)std::sin(ang);
        }
        for (int c = 0; c < kRopeLoRows; ++c) {
            double ang = (double)c * w;
            lo[(size_t)c * kRopeRowFloats + i] = (float)std::cos(ang);
            lo[(size_t)c * kRopeRowFloats + half + i] = (float)std::sin(ang);
        }
    }
}

std::string check_config(const hsq_config* c) {
    if (!c) return "config is NULL";
    if (c->head_dim != kDim) return "head_dim must be 128";
    if (c->n_q_heads < 1 || c->n_kv_heads < 1) return "head counts must be positive";
    if (c->n_q_heads % c->n_kv_heads) return "n_q_heads must be a multiple of n_kv_heads";
    if (c->group_n != 8 && c->group_n != 16) return "group_n must be 8 or 16";
    if (c->beta < 1 || c->beta > HSQ_MAX_BETA) return "beta must be in [1, 512]";
    if (c->bits_l1l3 != 4 || c->bits_l2 != 3) return "bits must be 4 (L1/L3) and 3 (L2)";
    if (!(c->rope_theta > 0.0)) return "rope_theta must be positive";
    if (c->max_batch < 1 || c->max_ctx < 1 || c->max_l1 < 0) return "capacities must be positive";
    if (c->max_pos < c->max_ctx || c->max_pos > (1 << 24)) return "max_pos must be in [max_ctx, 2^24]";
    if ((long long)c->max_ctx > (1LL << 24)) return "max_ctx too large";
    if ((c->max_ctx + c->group_n - 1) / c->group_n > 32768) return "more than 32768 groups per sequence";
    if (c->n_splits < 0 || c->n_splits > HSQ_MAX_SPLITS) return "n_splits must be in [0, 16]";
    if (c->l1_sinks < 0 || c->l1_recent < 0) return "l1_sinks and l1_recent must be >= 0";
    if (c->l1_recent > 0 && (long long)c->l1_sinks + c->l1_recent > c->max_l1)
        return "l1_sinks + l1_recent must fit max_l1";
    if (c->route_max != 0 && c->route_max != 1) return "route_max must be 0 or 1";
    if (c->codec != HSQ_CODEC_TQ && c->codec != HSQ_CODEC_PLAIN) return "codec must be HSQ_CODEC_TQ or HSQ_CODEC_PLAIN";
    if (c->route_per_head != 0 && c->route_per_head != 1) return "route_per_head must be 0 or 1";
    if (c->route_per_head && c->route_max) return "route_per_head and route_max exclude each other";
    if (c->qjl != 0 && c->qjl != 1) return "qjl must be 0 or 1";
    if (c->qjl && c->codec != HSQ_CODEC_TQ) return "qjl (TQ-QKV) needs the TurboQuant codec";
    if (c->hot_slots != 0) {
        if (c->hot_slots < 16 || c->hot_slots > hsq::kMaxHotSlots || (c->hot_slots & (c->hot_slots - 1)))
            return "hot_slots must be 0 or a power of two in [16, 1024]";
        if (c->codec != HSQ_CODEC_TQ || c->qjl || c->route_per_head)
            return "hot_slots needs codec HSQ_CODEC_TQ, qjl 0 and route_per_head 0";
    }
    if (c->overlap_launch != 0 && c->overlap_launch != 1) return "overlap_launch must be 0 or 1";
    return "";
}

std::string check_cache_shape(const hsq_config* cfg, const hsq_cache* c) {
    if (!c) return "cache is NULL";
    if (c->B < 1 || c->B > cfg->max_batch) return "cache B out of range";
    if (c->T < 1 || c->T > cfg->max_ctx) return "cache T out of range";
    if (c->t_cap != 0 && (c->t_cap < c->T || c->t_cap > cfg->max_ctx)) return "cache t_cap out of range";
    if (!c->l1_kc || !c->l1_vc || !c->l1_kn || !c->l1_vn || !c->l1_pos || !c->l1_count)
        return "an L1 buffer is NULL";
    if (!c->l2_kc || !c->l2_vc || !c->l2_kn || !c->l2_vn || !c->l2_cnt) return "an L2 buffer is NULL";
    if (!c->l3) return "l3 is NULL";
    if ((uintptr_t)c->l3 & 15u) return "l3 must be 16-byte aligned";
    if (!c->l1_bitmap) return "l1_bitmap is NULL";
    if (!c->signs && cfg->codec != HSQ_CODEC_PLAIN) return "signs is NULL";
    if (cfg->qjl && (!c->qjl_s || !c->l1_qs || !c->l1_qn || !c->l3_qs || !c->l3_qn))
        return "a key-residual sketch buffer is NULL (cfg.qjl)";
    if (cfg->hot_slots && (!c->hot_rec || !c->hot_tag)) return "hot_rec or hot_tag is NULL (cfg.hot_slots)";
    if (cfg->hot_slots && (((uintptr_t)c->hot_rec | (uintptr_t)c->hot_tag) & 15u))
        return "hot_rec and hot_tag must be 16-byte aligned";
    return "";
}

unsigned fault_mask() { return g_fault.load(); }

void set_process_error(const std::string& s) {
    std::lock_guard<std::mutex> lk(g_err_mu);
    g_err = s;
}

const char* process_error() {
    std::lock_guard<std::mutex> lk(g_err_mu);
    return g_err.c_str();
}

}  // namespace hsq

extern "C" {

hsq_status hsq_codebook(int bits, int dim, double* centroids, double* boundaries) {
    if (!centroids || !boundaries) return HSQ_ERR_INVALID;
    return hsq::lloyd_max(bits, dim, centroids, boundaries) ? HSQ_OK : HSQ_ERR_INVALID;
}

hsq_status hsq_cache_sizes(const hsq_config* cfg, int B, int T, size_t bytes[HSQ_NBUF]) {
    if (!bytes || !hsq::check_config(cfg).empty()) return HSQ_ERR_INVALID;
    if (B < 1 || B > cfg->max_batch || T < 1 || T > cfg->max_ctx) return HSQ_ERR_INVALID;
    const size_t H = cfg->n_kv_heads, L1 = cfg->max_l1, N = cfg->group_n;
    const size_t G = hsq::groups_of(T, cfg->group_n);
    bytes[HSQ_BUF_L1_KC] = B * H * L1 * 64;
    bytes[HSQ_BUF_L1_VC] = B * H * L1 * 64;
    bytes[HSQ_BUF_L1_KN] = B * H * L1 * 4;
    bytes[HSQ_BUF_L1_VN] = B * H * L1 * 4;
    bytes[HSQ_BUF_L1_POS] = B * L1 * 4;
    bytes[HSQ_BUF_L1_COUNT] = (size_t)B * 4;
    bytes[HSQ_BUF_L2_KC] = B * H * G * 48;
    bytes[HSQ_BUF_L2_VC] = B * H * G * 48;
    bytes[HSQ_BUF_L2_KN] = B * H * G * 4;
    bytes[HSQ_BUF_L2_VN] = B * H * G * 4;
    bytes[HSQ_BUF_L2_CNT] = B * G;
    bytes[HSQ_BUF_L3] = B * H * G * hsq::record_bytes((int)N);
    bytes[HSQ_BUF_L1_BITMAP] = (size_t)B * hsq::bitmap_words(T) * 4;
    const size_t Hs = cfg->route_per_head ? (size_t)cfg->n_q_heads : H;  // selection rows per sequence
    bytes[HSQ_BUF_STAGING] = B * Hs * (size_t)cfg->beta * hsq::record_bytes((int)N);
    bytes[HSQ_BUF_WIN_KV] = B * H * (size_t)cfg->l1_recent * 2 * hsq::kDim * 4;
    bytes[HSQ_BUF_GSUM] = cfg->l1_recent > 0 ? B * H * (size_t)hsq::kGsumFloats * 4 : 0;
    const size_t q = cfg->qjl ? 1 : 0;  // key-residual sketches: 16 B of bits + a float norm per key
    bytes[HSQ_BUF_L1_QS] = q * B * H * L1 * 16;
    bytes[HSQ_BUF_L1_QN] = q * B * H * L1 * 4;
    bytes[HSQ_BUF_L3_QS] = q * B * H * G * N * 16;
    bytes[HSQ_BUF_L3_QN] = q * B * H * G * N * 4;
    const size_t hs = (size_t)cfg->hot_slots;  // hot-group table: records and tags
    bytes[HSQ_BUF_HOT_REC] = B * H * hs * hsq::record_bytes((int)N);
    bytes[HSQ_BUF_HOT_TAG] = B * H * hs * 4;
    return HSQ_OK;
}

hsq_status hsq_debug_set_fault(unsigned mask) {
    hsq::g_fault.store(mask);
    return HSQ_OK;
}

const char* hsq_version(void) { return "hsq-gb300 0.1"; }

}  // extern "C"
