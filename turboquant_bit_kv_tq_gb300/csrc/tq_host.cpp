// Host side of the library: configuration checks, page layout, the seeded
// parameter tables (rotation signs, QJL matrix, Lloyd-Max codebooks) and the
// handle / error-word entry points of tq_kv.h.

#include <math.h>
#include <string.h>

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <map>
#include <mutex>
#include <new>
#include <utility>
#include <vector>

#include "tq_internal.h"

namespace tq {

// ---------------------------------------------------------------- layout
tq_status compute_layout(const tq_cache_config& c, Layout* lay) {
    if (c.head_dim != 128 && c.head_dim != 256) return TQ_ERR_UNSUPPORTED;
    if (c.block_size != kBlock) return TQ_ERR_UNSUPPORTED;
    if (c.k_bits < 2 || c.k_bits > 4 || c.v_bits < 2 || c.v_bits > 4) return TQ_ERR_UNSUPPORTED;
    if (c.v_mode != TQ_V_MSE && c.v_mode != TQ_V_G32) return TQ_ERR_UNSUPPORTED;
    // group-32 values pack 2 or 4 bits per coordinate ([Hub] step 4)
    if (c.v_mode == TQ_V_G32 && c.v_bits != 2 && c.v_bits != 4) return TQ_ERR_UNSUPPORTED;
    if (c.k_qjl != 0 && c.k_qjl != 1) return TQ_ERR_INVALID_ARG;
    if (c.k_codebook != TQ_CODEBOOK_LLOYD && c.k_codebook != TQ_CODEBOOK_UNIFORM) return TQ_ERR_INVALID_ARG;
    if (c.v_codebook != TQ_CODEBOOK_LLOYD && c.v_codebook != TQ_CODEBOOK_UNIFORM) return TQ_ERR_INVALID_ARG;
    if (c.v_mode == TQ_V_G32 && c.v_codebook != TQ_CODEBOOK_LLOYD) return TQ_ERR_INVALID_ARG;
    if (c.num_kv_heads < 1 || c.num_q_heads < c.num_kv_heads || c.num_q_heads % c.num_kv_heads) return TQ_ERR_INVALID_ARG;
    {
        const int G = c.num_q_heads / c.num_kv_heads;  // grouped query heads per KV head
        if (G > 16 || (G > 4 && G % 4)) return TQ_ERR_UNSUPPORTED;
    }
    if (c.num_blocks < 1 || c.max_batch < 1 || c.max_blocks_per_seq < 1 || c.split_blocks < 1 || c.tail_cap < 0)
        return TQ_ERR_INVALID_ARG;
    Layout L;
    const int d = c.head_dim;
    L.d = d;
    L.k_bits = c.k_bits;
    L.v_bits = c.v_bits;
    L.k_qjl = c.k_qjl;
    L.v_mode = c.v_mode;
    L.k_code_row = d * c.k_bits / 8;
    L.k_sign_row = d / 8;
    L.v_code_row = d * c.v_bits / 8;
    L.v_meta_row = c.v_mode == TQ_V_MSE ? 2 : 4 * (d / 32);
    int off = 0;
    L.k_codes = off;
    off += kBlock * L.k_code_row;
    L.k_signs = off;
    off += c.k_qjl ? kBlock * L.k_sign_row : 0;
    L.k_norm = off;
    off += kBlock * 2;
    L.k_rnorm = off;
    off += c.k_qjl ? kBlock * 2 : 0;
    L.v_codes = off;
    off += kBlock * L.v_code_row;
    L.v_meta = off;
    off += kBlock * L.v_meta_row;
    L.page_bytes = off;
    *lay = L;
    return TQ_OK;
}

Splits compute_splits(const tq_cache_config& c) {
    Splits s;
    s.n_chunks = (c.max_blocks_per_seq + c.split_blocks - 1) / c.split_blocks;
    s.n_splits = s.n_chunks + (c.tail_cap > 0 ? 1 : 0);
    return s;
}

static size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

ParamsLayout params_layout(const tq_cache_config& c) {
    const size_t d = c.head_dim;
    ParamsLayout p;
    size_t off = 0;
    p.signs = off;
    off = up256(off + d * 4);
    p.s_f32 = off;
    off = up256(off + d * d * 4);
    p.st_f32 = off;
    off = up256(off + d * d * 4);
    p.s_bf16 = off;
    off = up256(off + d * d * 2);
    p.st_bf16 = off;
    off = up256(off + d * d * 2);
    p.k_cent = off;
    off = up256(off + kMaxLevels * 4);
    p.k_bound = off;
    off = up256(off + kMaxLevels * 4);
    p.v_cent = off;
    off = up256(off + kMaxLevels * 4);
    p.v_bound = off;
    off = up256(off + kMaxLevels * 4);
    p.k_walsh = off;
    off = up256(off + 9 * 4);
    p.v_walsh = off;
    off = up256(off + 9 * 4);
    p.t_hi = off;
    off = up256(off + d * d * 2);
    p.t_lo = off;
    off = up256(off + d * d * 2);
    p.err = off;
    off = up256(off + 4);
    p.total = off;
    return p;
}

DecodeGeom decode_geom(const tq_cache_config& c) {
    DecodeGeom g;
    const int G = c.num_q_heads / c.num_kv_heads;
    // head groups of at most 4 query heads (one n-tile: the warp-specialized
    // split kernel's consumers hold one n-tile of value accumulators)
    g.hc = G <= 4 ? G : 4;
    g.nhg = G / g.hc;
    g.nth = (g.hc + 3) / 4;
    g.npk = 1 << (c.k_bits - 1);
    g.npl = g.npk + (c.k_qjl ? 1 : 0);
    g.n_cols = (kPieces * 4 * g.nth + 15) / 16 * 16;
    g.bimg_bytes = g.n_cols * g.npl * c.head_dim;
    return g;
}

WorkspaceLayout workspace_layout(const tq_cache_config& c) {
    const Splits s = compute_splits(c);
    const DecodeGeom gm = decode_geom(c);
    const size_t bh = size_t(c.max_batch) * c.num_q_heads, d = c.head_dim;
    WorkspaceLayout w;
    size_t off = 0;
    w.bimg = off;
    off = up256(off + size_t(c.max_batch) * c.num_kv_heads * gm.nhg * gm.bimg_bytes);
    w.cst = off;
    off = up256(off + bh * 4 * 4);
    w.acc = off;
    off = up256(off + bh * s.n_splits * d * 4);
    w.ml = off;
    off = up256(off + bh * s.n_splits * 2 * 4);
    w.ext = off;  // 4 x [B] int32, 4 int32 counts, [B] int4 query blocks
    off = up256(off + size_t(c.max_batch) * 4 * 4 + 16 + size_t(c.max_batch) * 16);
    w.total = off;
    return w;
}

// ------------------------------------------------------------ parameters
// SplitMix64 (Steele, Lea & Flood, OOPSLA 2014): the state advances by the
// golden-ratio increment and each output is a bijective mix of the state.
struct SplitMix64 {
    uint64_t state;
    explicit SplitMix64(uint64_t seed) : state(seed) {}
    uint64_t next() {
        state += 0x9E3779B97F4A7C15ull;
        uint64_t z = state;
        z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
        z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
        return z ^ (z >> 31);
    }
    // (x >> 11 + 1/2) * 2^-53: a double strictly inside (0, 1)
    double uniform() { return ((double)(next() >> 11) + 0.5) * 0x1.0p-53; }
};

// Round a double to the nearest bfloat16 (ties to even), returning its bits.
static uint16_t bf16_bits_from_double(double x) {
    uint64_t u;
    memcpy(&u, &x, 8);
    const uint64_t dropped = 52 - 7;  // fraction bits a bf16 does not keep
    u += ((1ull << (dropped - 1)) - 1) + ((u >> dropped) & 1);
    u &= ~((1ull << dropped) - 1);
    double r;
    memcpy(&r, &u, 8);
    float f = (float)r;  // exact: r has at most 8 significant bits
    uint32_t b;
    memcpy(&b, &f, 4);
    return (uint16_t)(b >> 16);
}

// fp16 bit pattern of a float, round to nearest even (finite inputs of
// magnitude below 65504; subnormal results included)
static uint16_t f16_bits(float f) {
    uint32_t x;
    memcpy(&x, &f, 4);
    const uint16_t sign = (uint16_t)((x >> 16) & 0x8000u);
    x &= 0x7FFFFFFFu;
    if (x >= 0x477FF000u) return sign | 0x7C00u;  // rounds past the largest fp16: infinity
    if (x < 0x38800000u) {                         // below 2^-14: a multiple of 2^-24
        const float m = nearbyintf(fabsf(f) * 16777216.0f);
        return sign | (uint16_t)m;                  // (m = 1024 encodes 2^-14 exactly)
    }
    return sign | (uint16_t)((x + 0x00000FFFu + ((x >> 13) & 1u) - 0x38000000u) >> 13);
}

static float f16_to_float(uint16_t h) {
    const uint32_t e = (h >> 10) & 31u, m = h & 1023u;
    const float v = e == 0 ? ldexpf((float)m, -24) : ldexpf((float)(m | 1024u), (int)e - 25);
    return (h & 0x8000u) ? -v : v;
}

static float bf16_to_float(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

// Rotation diagonal: sign -1 when the top bit of the i-th draw is set.
static void make_signs(int d, uint64_t seed, std::vector<float>& signs) {
    SplitMix64 g(seed);
    signs.resize(d);
    for (int i = 0; i < d; ++i) signs[i] = (g.next() >> 63) ? -1.f : 1.f;
}

// QJL matrix: N(0,1) entries in row-major order by Box-Muller on consecutive
// draw pairs (cosine branch first), each rounded to bf16.
static void make_qjl(int d, uint64_t seed, std::vector<uint16_t>& s) {
    SplitMix64 g(seed);
    s.resize((size_t)d * d);
    for (size_t p = 0; p < s.size() / 2; ++p) {
        const double u1 = g.uniform(), u2 = g.uniform();
        const double radius = sqrt(-2.0 * log(u1));
        s[2 * p] = bf16_bits_from_double(radius * cos(2.0 * M_PI * u2));
        s[2 * p + 1] = bf16_bits_from_double(radius * sin(2.0 * M_PI * u2));
    }
}

// Gauss-Legendre nodes and weights on [-1, 1] (Newton iteration on the
// three-term Legendre recurrence).
static void gauss_legendre(int n, std::vector<double>& x, std::vector<double>& w) {
    x.assign(n, 0.0);
    w.assign(n, 0.0);
    for (int i = 0; i < (n + 1) / 2; ++i) {
        double z = cos(M_PI * (i + 0.75) / (n + 0.5)), dp = 1.0;
        for (int it = 0; it < 100; ++it) {
            double p0 = 1.0, p1 = 0.0;
            for (int j = 1; j <= n; ++j) {
                const double p2 = p1;
                p1 = p0;
                p0 = ((2.0 * j - 1.0) * z * p1 - (j - 1.0) * p2) / j;
            }
            dp = n * (z * p0 - p1) / (z * z - 1.0);
            const double dz = p0 / dp;
            z -= dz;
            if (fabs(dz) < 1e-16) break;
        }
        x[i] = -z;
        x[n - 1 - i] = z;
        w[i] = w[n - 1 - i] = 2.0 / ((1.0 - z * z) * dp * dp);
    }
}

// Density of one coordinate of a uniform unit vector in R^d:
// f(t) = C (1 - t^2)^((d-3)/2), C = Gamma(d/2) / (sqrt(pi) Gamma((d-1)/2)).
struct SphereDensity {
    int d;
    double C;
    std::vector<double> gx, gw;
    explicit SphereDensity(int d_) : d(d_) {
        C = exp(lgamma(0.5 * d) - lgamma(0.5 * (d - 1))) / sqrt(M_PI);
        gauss_legendre(48, gx, gw);
    }
    double f(double t) const { return C * exp(0.5 * (d - 3) * log1p(-t * t)); }
    // P(a < T < b): composite Gauss-Legendre on 32 panels
    double mass(double a, double b) const {
        const int panels = 32;
        const double h = (b - a) / panels;
        double s = 0.0;
        for (int p = 0; p < panels; ++p) {
            const double lo = a + p * h, mid = lo + 0.5 * h;
            for (size_t k = 0; k < gx.size(); ++k) s += gw[k] * f(mid + 0.5 * h * gx[k]);
        }
        return 0.5 * h * s;
    }
    // integral of t f(t) over (a, b): C/(d-1) [(1-a^2)^((d-1)/2) - (1-b^2)^((d-1)/2)]
    double moment(double a, double b) const {
        const double e = 0.5 * (d - 1);
        return C / (d - 1) * (exp(e * log1p(-a * a)) - exp(e * log1p(-b * b)));
    }
};

// Expansion of a symmetric codebook over XOR bit-planes: with chi_S(i) =
// (-1)^popcount(i & S), c[i] = sum_S chat_S chi_S(i), chat_S = mean_i c[i] chi_S(i);
// symmetry (c[L-1-i] = -c[i]) leaves only odd |S|.  Writing chi_S = 1 - 2 u_S,
// u_S = XOR of the bits of i in S:  c[i] = alpha + sum_S beta_S u_S(i) with
// alpha = sum_S chat_S, beta_S = -2 chat_S.  out = {alpha, beta_S...} in the
// order of plane_subset().
// A uniform codebook c[i] = step (i - (L-1)/2) is linear in the bits of i, so
// every multi-bit term is zero: those are set to exactly zero (single_bits).
static void walsh_planes(const std::vector<double>& c, int bits, float* out, bool single_bits = false) {
    const int L = 1 << bits, planes = 1 << (bits - 1);
    double alpha = 0.0;
    for (int pi = 0; pi < planes; ++pi) {
        const int S = plane_subset(bits, pi);
        double chat = 0.0;
        for (int i = 0; i < L; ++i) chat += (__builtin_popcount(i & S) & 1) ? -c[i] : c[i];
        chat /= L;
        if (single_bits && __builtin_popcount(S) > 1) chat = 0.0;
        alpha += chat;
        out[1 + pi] = (float)(-2.0 * chat);
    }
    out[0] = (float)alpha;
}

static void lloyd_max_sphere(int d, int bits, std::vector<double>& c, std::vector<double>& b, double* mse) {
    const int L = 1 << bits;
    const SphereDensity dens(d);
    const double sigma = 1.0 / sqrt((double)d);
    c.resize(L);
    b.resize(L - 1);
    for (int i = 0; i < L; ++i) c[i] = std::max(-0.999, std::min(0.999, sigma * (-2.0 + 4.0 * (i + 0.5) / L)));
    std::vector<double> edges(L + 1), next(L);
    for (int it = 0; it < 20000; ++it) {
        edges[0] = -1.0;
        edges[L] = 1.0;
        for (int i = 0; i + 1 < L; ++i) edges[i + 1] = 0.5 * (c[i] + c[i + 1]);
        // even density: compute the lower half and mirror
        for (int i = 0; i < L / 2; ++i) next[i] = dens.moment(edges[i], edges[i + 1]) / dens.mass(edges[i], edges[i + 1]);
        for (int i = 0; i < L / 2; ++i) next[L - 1 - i] = -next[i];
        double moved = 0.0;
        for (int i = 0; i < L; ++i) moved = std::max(moved, fabs(next[i] - c[i]));
        c = next;
        if (moved < 1e-15) break;
    }
    for (int i = 0; i + 1 < L; ++i) b[i] = 0.5 * (c[i] + c[i + 1]);
    if (mse) {
        double s = 0.0;
        for (int i = 0; i < L; ++i) {
            const double lo = i == 0 ? -1.0 : b[i - 1], hi = i == L - 1 ? 1.0 : b[i];
            s += dens.mass(lo, hi) * c[i] * c[i];
        }
        *mse = 1.0 - d * s;
    }
}

}  // namespace tq

using namespace tq;

namespace tq {
static thread_local char g_cuda_msg[384] = "";
tq_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return TQ_OK;
    snprintf(g_cuda_msg, sizeof g_cuda_msg, "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
    return TQ_ERR_CUDA;
}
tq_status driver_failure(const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_cuda_msg, sizeof g_cuda_msg, fmt, ap);
    va_end(ap);
    return TQ_ERR_CUDA;
}
tq_status cuda_status_detail(cudaError_t e, const char* fmt, ...) {
    if (cuda_status(e) == TQ_OK) return TQ_OK;
    const size_t n = strlen(g_cuda_msg);
    if (n + 3 < sizeof g_cuda_msg) {
        g_cuda_msg[n] = ' ';
        g_cuda_msg[n + 1] = '(';
        va_list ap;
        va_start(ap, fmt);
        vsnprintf(g_cuda_msg + n + 2, sizeof g_cuda_msg - n - 3, fmt, ap);
        va_end(ap);
        const size_t m = strlen(g_cuda_msg);
        if (m + 1 < sizeof g_cuda_msg) {
            g_cuda_msg[m] = ')';
            g_cuda_msg[m + 1] = 0;
        }
    }
    return TQ_ERR_CUDA;
}

// Per-device launch state, shared by every host thread: each device's SM
// count, and the dynamic shared-memory limit already granted to each kernel on
// each device (cudaFuncSetAttribute acts on the calling thread's current
// device).  One mutex guards both; a lookup costs one uncontended lock.
static std::mutex g_dev_mu;
static std::vector<int> g_dev_sms;
static std::map<std::pair<int, const void*>, int> g_dev_smem;

static tq_status current_device(int* dev) {
    const tq_status st = cuda_status(cudaGetDevice(dev));
    return st != TQ_OK ? st : (*dev < 0 ? TQ_ERR_CUDA : TQ_OK);
}

tq_status device_sms(int* sms) {
    int dev = 0;
    const tq_status st = current_device(&dev);
    if (st != TQ_OK) return st;
    std::lock_guard<std::mutex> lock(g_dev_mu);
    if ((int)g_dev_sms.size() <= dev) g_dev_sms.resize(dev + 1, 0);
    if (g_dev_sms[dev] <= 0) {
        int n = 0;
        const tq_status a = cuda_status(cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev));
        if (a != TQ_OK) return a;
        if (n <= 0) return TQ_ERR_CUDA;
        g_dev_sms[dev] = n;
    }
    *sms = g_dev_sms[dev];
    return TQ_OK;
}

tq_status ensure_dynamic_smem(const void* func, int bytes, const char* name) {
    int dev = 0;
    const tq_status st = current_device(&dev);
    if (st != TQ_OK) return st;
    std::lock_guard<std::mutex> lock(g_dev_mu);
    int& granted = g_dev_smem[std::make_pair(dev, func)];
    if (granted >= bytes) return TQ_OK;
    const tq_status a = cuda_status_detail(
        cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes),
        "%s dynamic shared memory %d on device %d", name, bytes, dev);
    if (a == TQ_OK) granted = bytes;
    return a;
}
}  // namespace tq

extern "C" {

const char* tq_last_cuda_error(void) { return tq::g_cuda_msg; }

const char* tq_status_string(tq_status s) {
    switch (s) {
        case TQ_OK: return "ok";
        case TQ_ERR_INVALID_ARG: return "invalid argument";
        case TQ_ERR_UNSUPPORTED: return "unsupported configuration (d must be 128/256, bits 2..4, block 16)";
        case TQ_ERR_BUFFER_TOO_SMALL: return "buffer too small";
        case TQ_ERR_CUDA: return "CUDA runtime error";
        case TQ_ERR_MISALIGNED: return "device pointer not 16-byte aligned";
        default: return "unknown status";
    }
}

// Distortion-optimal uniform grid c[i] = step k_i, k_i = i - (L-1)/2, with
// midpoint boundaries.  The distortion's derivative in the step is
// -2 g(step), g = sum_i k_i M_i - step sum_i k_i^2 P_i over the midpoint cells
// (M, P: first moment and mass of a cell; the boundary terms cancel because
// the integrand is continuous at a midpoint).  g > 0 for a tiny step and
// g < 0 once the outer centroids pass +-1; the optimum is its root, found by
// bisection to machine precision.
static void uniform_sphere(int d, int bits, std::vector<double>& c, std::vector<double>& b, double* mse) {
    const int L = 1 << bits;
    const SphereDensity dens(d);
    std::vector<double> k(L), edges(L + 1), P(L), M(L);
    for (int i = 0; i < L; ++i) k[i] = i - 0.5 * (L - 1);
    auto cells = [&](double st) {
        edges[0] = -1.0;
        edges[L] = 1.0;
        for (int i = 0; i + 1 < L; ++i) edges[i + 1] = std::max(-1.0, std::min(1.0, st * (k[i] + 0.5)));
        for (int i = 0; i < L; ++i) {
            P[i] = dens.mass(edges[i], edges[i + 1]);
            M[i] = dens.moment(edges[i], edges[i + 1]);
        }
    };
    auto g = [&](double st) {
        cells(st);
        double num = 0.0, den = 0.0;
        for (int i = 0; i < L; ++i) {
            num += k[i] * M[i];
            den += k[i] * k[i] * P[i];
        }
        return num - st * den;
    };
    double lo = 1e-6 / sqrt((double)d), hi = 2.0 / (L - 1);
    for (int it = 0; it < 200 && hi - lo > 1e-16 * hi; ++it) {
        const double mid = 0.5 * (lo + hi);
        (g(mid) > 0.0 ? lo : hi) = mid;
    }
    const double step = 0.5 * (lo + hi);
    c.resize(L);
    b.resize(L - 1);
    for (int i = 0; i < L; ++i) c[i] = step * k[i];
    for (int i = 0; i + 1 < L; ++i) b[i] = 0.5 * (c[i] + c[i + 1]);
    if (mse) {
        // d E[(t - Q t)^2] = 1 - d sum_i (2 c_i M_i - c_i^2 P_i), E[t^2] = 1/d
        cells(step);
        double s = 0.0;
        for (int i = 0; i < L; ++i) s += 2.0 * c[i] * M[i] - c[i] * c[i] * P[i];
        *mse = 1.0 - d * s;
    }
}

static void make_codebook(int kind, int d, int bits, std::vector<double>& c, std::vector<double>& b) {
    if (kind == TQ_CODEBOOK_UNIFORM)
        uniform_sphere(d, bits, c, b, nullptr);
    else
        lloyd_max_sphere(d, bits, c, b, nullptr);
}

tq_status tq_make_uniform_codebook(int d, int bits, double* centroids, double* boundaries, double* mse) {
    if (d < 3 || bits < 1 || bits > 8 || !centroids || !boundaries) return TQ_ERR_INVALID_ARG;
    std::vector<double> c, b;
    uniform_sphere(d, bits, c, b, mse);
    std::copy(c.begin(), c.end(), centroids);
    std::copy(b.begin(), b.end(), boundaries);
    return TQ_OK;
}

tq_status tq_make_codebook(int d, int bits, double* centroids, double* boundaries, double* mse) {
    if (d < 3 || bits < 1 || bits > 8 || !centroids || !boundaries) return TQ_ERR_INVALID_ARG;
    std::vector<double> c, b;
    lloyd_max_sphere(d, bits, c, b, mse);
    std::copy(c.begin(), c.end(), centroids);
    std::copy(b.begin(), b.end(), boundaries);
    return TQ_OK;
}

tq_status tq_make_rotation_signs(int d, uint64_t seed, float* signs) {
    if (d < 2 || !signs) return TQ_ERR_INVALID_ARG;
    std::vector<float> s;
    make_signs(d, seed, s);
    std::copy(s.begin(), s.end(), signs);
    return TQ_OK;
}

tq_status tq_make_qjl_matrix(int d, uint64_t seed, uint16_t* s_bf16) {
    if (d < 2 || (d & 1) || !s_bf16) return TQ_ERR_INVALID_ARG;
    std::vector<uint16_t> s;
    make_qjl(d, seed, s);
    std::copy(s.begin(), s.end(), s_bf16);
    return TQ_OK;
}

tq_status tq_cache_sizes(const tq_cache_config* cfg, size_t* page_bytes, size_t* cache_bytes, size_t* params_bytes,
                         size_t* workspace_bytes) {
    if (!cfg) return TQ_ERR_INVALID_ARG;
    Layout lay;
    const tq_status st = compute_layout(*cfg, &lay);
    if (st != TQ_OK) return st;
    if (page_bytes) *page_bytes = lay.page_bytes;
    if (cache_bytes) *cache_bytes = (size_t)cfg->num_blocks * cfg->num_kv_heads * lay.page_bytes;
    if (params_bytes) *params_bytes = params_layout(*cfg).total;
    if (workspace_bytes) *workspace_bytes = workspace_layout(*cfg).total;
    return TQ_OK;
}

tq_status tq_cache_create(const tq_cache_config* cfg, void* params_dev, void* workspace_dev, void* stream,
                          tq_cache** out) {
    if (!cfg || !params_dev || !workspace_dev || !out) return TQ_ERR_INVALID_ARG;
    *out = nullptr;
    Layout lay;
    tq_status st = compute_layout(*cfg, &lay);
    if (st != TQ_OK) return st;
    if (((uintptr_t)params_dev & 255) || ((uintptr_t)workspace_dev & 15)) return TQ_ERR_MISALIGNED;
    tq_cache* h = new (std::nothrow) tq_cache();
    if (!h) return TQ_ERR_INVALID_ARG;
    h->cfg = *cfg;
    h->lay = lay;
    h->splits = compute_splits(*cfg);
    const int d = cfg->head_dim;
    make_signs(d, cfg->seed_rot, h->signs);
    make_qjl(d, cfg->seed_qjl, h->s_bf16);
    make_codebook(cfg->k_codebook, d, cfg->k_bits, h->k_cent, h->k_bound);
    if (cfg->v_mode == TQ_V_MSE) make_codebook(cfg->v_codebook, d, cfg->v_bits, h->v_cent, h->v_bound);

    // stage the device tables on the host, then one copy
    const ParamsLayout pl = params_layout(*cfg);
    std::vector<uint8_t> img(pl.total, 0);
    float* signs = (float*)(img.data() + pl.signs);
    float* s32 = (float*)(img.data() + pl.s_f32);
    float* st32 = (float*)(img.data() + pl.st_f32);
    uint16_t* s16 = (uint16_t*)(img.data() + pl.s_bf16);
    uint16_t* st16 = (uint16_t*)(img.data() + pl.st_bf16);
    for (int i = 0; i < d; ++i) signs[i] = h->signs[i];
    for (int j = 0; j < d; ++j)
        for (int i = 0; i < d; ++i) {
            const uint16_t bits = h->s_bf16[(size_t)j * d + i];
            s16[(size_t)j * d + i] = bits;
            st16[(size_t)i * d + j] = bits;
            s32[(size_t)j * d + i] = bf16_to_float(bits);
            st32[(size_t)i * d + j] = bf16_to_float(bits);
        }
    auto put = [&](size_t off, const std::vector<double>& v) {
        float* p = (float*)(img.data() + off);
        for (size_t i = 0; i < v.size(); ++i) p[i] = (float)v[i];
        for (size_t i = v.size(); i < (size_t)kMaxLevels; ++i) p[i] = INFINITY;
    };
    put(pl.k_cent, h->k_cent);
    put(pl.k_bound, h->k_bound);
    put(pl.v_cent, h->v_cent);
    put(pl.v_bound, h->v_bound);
    walsh_planes(h->k_cent, cfg->k_bits, (float*)(img.data() + pl.k_walsh), cfg->k_codebook == TQ_CODEBOOK_UNIFORM);
    {
        // T = S D H / sqrt(d) in fp64 (H_ki = (-1)^popcount(k & i)), split
        // into fp16 high and low parts
        uint16_t* thi = (uint16_t*)(img.data() + pl.t_hi);
        uint16_t* tlo = (uint16_t*)(img.data() + pl.t_lo);
        std::vector<double> row(d);
        const double inv = 1.0 / sqrt((double)d);
        for (int j = 0; j < d; ++j) {
            for (int k = 0; k < d; ++k) row[k] = (double)bf16_to_float(h->s_bf16[(size_t)j * d + k]) * h->signs[k];
            // row <- row H (Sylvester H is symmetric: a Walsh-Hadamard transform)
            for (int len = 1; len < d; len <<= 1)
                for (int k = 0; k < d; k += 2 * len)
                    for (int u = k; u < k + len; ++u) {
                        const double a = row[u], b = row[u + len];
                        row[u] = a + b;
                        row[u + len] = a - b;
                    }
            for (int i = 0; i < d; ++i) {
                const double t = row[i] * inv;
                const uint16_t hb = f16_bits((float)t);
                thi[(size_t)j * d + i] = hb;
                tlo[(size_t)j * d + i] = f16_bits((float)(t - (double)f16_to_float(hb)));
            }
        }
    }
    if (cfg->v_mode == TQ_V_MSE)
        walsh_planes(h->v_cent, cfg->v_bits, (float*)(img.data() + pl.v_walsh), cfg->v_codebook == TQ_CODEBOOK_UNIFORM);
    cudaStream_t s = (cudaStream_t)stream;
    if (cudaMemcpyAsync(params_dev, img.data(), img.size(), cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
        delete h;
        return TQ_ERR_CUDA;
    }
    uint8_t* base = (uint8_t*)params_dev;
    h->dp.signs = (const float*)(base + pl.signs);
    h->dp.s_f32 = (const float*)(base + pl.s_f32);
    h->dp.st_f32 = (const float*)(base + pl.st_f32);
    h->dp.s_bf16 = (const uint16_t*)(base + pl.s_bf16);
    h->dp.st_bf16 = (const uint16_t*)(base + pl.st_bf16);
    h->dp.k_cent = (const float*)(base + pl.k_cent);
    h->dp.k_bound = (const float*)(base + pl.k_bound);
    h->dp.v_cent = (const float*)(base + pl.v_cent);
    h->dp.v_bound = (const float*)(base + pl.v_bound);
    h->dp.k_walsh = (const float*)(base + pl.k_walsh);
    h->dp.v_walsh = (const float*)(base + pl.v_walsh);
    h->dp.t_hi = (const uint16_t*)(base + pl.t_hi);
    h->dp.t_lo = (const uint16_t*)(base + pl.t_lo);
    h->dp.err = (uint32_t*)(base + pl.err);
    const WorkspaceLayout wl = workspace_layout(*cfg);
    uint8_t* ws = (uint8_t*)workspace_dev;
    h->geom = decode_geom(*cfg);
    h->ws_bimg = (uint8_t*)(ws + wl.bimg);
    h->ws_cst = (float*)(ws + wl.cst);
    h->ws_acc = (float*)(ws + wl.acc);
    h->ws_ml = (float*)(ws + wl.ml);
    h->ws_ext = (int32_t*)(ws + wl.ext);
    *out = h;
    return TQ_OK;
}

tq_status tq_cache_destroy(tq_cache* cache) {
    delete cache;
    return TQ_OK;
}

tq_status tq_cache_export_params(const tq_cache* c, float* signs, uint16_t* qjl_bf16, double* k_centroids,
                                 double* k_boundaries, double* v_centroids, double* v_boundaries) {
    if (!c) return TQ_ERR_INVALID_ARG;
    if (signs) std::copy(c->signs.begin(), c->signs.end(), signs);
    if (qjl_bf16) std::copy(c->s_bf16.begin(), c->s_bf16.end(), qjl_bf16);
    if (k_centroids) std::copy(c->k_cent.begin(), c->k_cent.end(), k_centroids);
    if (k_boundaries) std::copy(c->k_bound.begin(), c->k_bound.end(), k_boundaries);
    if (v_centroids) std::copy(c->v_cent.begin(), c->v_cent.end(), v_centroids);
    if (v_boundaries) std::copy(c->v_bound.begin(), c->v_bound.end(), v_boundaries);
    return TQ_OK;
}

tq_status tq_set_profile_events(tq_cache* c, int kernel, void* start_event, void* stop_event) {
    if (!c || kernel < 0 || kernel > 1 || ((start_event == nullptr) != (stop_event == nullptr))) return TQ_ERR_INVALID_ARG;
    c->prof_start[kernel] = start_event;
    c->prof_stop[kernel] = stop_event;
    return TQ_OK;
}

tq_status tq_get_device_error(const tq_cache* c, uint32_t* flags, void* stream) {
    if (!c || !flags) return TQ_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    uint32_t v = 0;
    if (cudaMemcpyAsync(&v, c->dp.err, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemsetAsync(c->dp.err, 0, 4, s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess)
        return TQ_ERR_CUDA;
    *flags = v;
    return TQ_OK;
}

}  // extern "C"
