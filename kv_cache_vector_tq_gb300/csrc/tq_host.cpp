// Host side of libtq: status codes, the offline Lloyd-Max codebook builder,
// Householder QR for the Haar rotation, context creation (operand tables in
// the layouts the kernels read), code layouts and the canonical unpacker.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <functional>
#include <thread>
#include <vector>

#include "tq_internal.h"

namespace tq {

static std::atomic<int> g_last_cuda_error{0};

tq_status set_cuda_error(cudaError_t e) {
  g_last_cuda_error.store((int)e);
  return TQ_ERR_CUDA;
}

int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return -1;
  }
  return dev;
}

int num_sms() {
  static PerDeviceValue cache;
  const int dev = current_device();
  const int n = cache.get(dev, [dev] {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      (void)cudaGetLastError();
      return -1;
    }
    return v;
  });
  return n > 0 ? n : 152;
}

cudaError_t smem_attr_once(PerDeviceValue& flag, const void* func, int bytes) {
  const int dev = current_device();
  if (dev < 0) return cudaErrorInvalidDevice;
  cudaError_t err = cudaSuccess;
  const int r = flag.get(dev, [&] {
    err = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    return err == cudaSuccess ? 1 : -1;
  });
  return r > 0 ? cudaSuccess : (err != cudaSuccess ? err : cudaErrorInvalidDevice);
}

int ctas_per_sm_once(PerDeviceValue& cache, const void* func, int threads, size_t smem) {
  const int dev = current_device();
  const int n = cache.get(dev, [&] {
    int v = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, func, threads, smem) != cudaSuccess) {
      (void)cudaGetLastError();
      return -1;
    }
    return v;
  });
  return n > 0 ? n : 1;
}

// Sum with Neumaier compensation, so the result does not depend on the order
// of the terms beyond the last bit.
struct KSum {
  double s = 0.0, c = 0.0;
  void add(double x) {
    double t = s + x;
    if (std::fabs(s) >= std::fabs(x))
      c += (s - t) + x;
    else
      c += (x - t) + s;
    s = t;
  }
  double value() const { return s + c; }
};

static void parallel_for(int n, int min_grain, const std::function<void(int, int)>& fn) {
  unsigned hw = std::thread::hardware_concurrency();
  int nt = (int)std::min<unsigned>(hw ? hw : 1, 16);
  if (n < 2 * min_grain || nt <= 1) {
    fn(0, n);
    return;
  }
  nt = std::min(nt, std::max(1, n / min_grain));
  std::vector<std::thread> th;
  int per = (n + nt - 1) / nt;
  for (int i = 0; i < nt; ++i) {
    int a = i * per, b = std::min(n, a + per);
    if (a >= b) break;
    th.emplace_back([=, &fn] { fn(a, b); });
  }
  for (auto& t : th) t.join();
}

// ---------------------------------------------------------------- codebook
// Density of one coordinate of a uniformly random unit vector in R^d
// ("TurboQuant 详解", section 关键洞察：先旋转), or its N(0, 1/d) limit.
static double coord_density(double x, int d, int density) {
  if (density == TQ_DENS_GAUSS) return std::sqrt(d / (2.0 * M_PI)) * std::exp(-0.5 * d * x * x);
  if (!(std::fabs(x) < 1.0)) return 0.0;
  double logc = std::lgamma(d / 2.0) - 0.5 * std::log(M_PI) - std::lgamma((d - 1) / 2.0);
  return std::exp(logc + ((d - 3) / 2.0) * std::log1p(-x * x));
}

static tq_status build_codebook(int d, int b, int density, int grid, int iters, tq_codebook* out) {
  const int K = 1 << b;
  const double sigma = 1.0 / std::sqrt((double)d);
  // grid over ±6σ; the Beta density has support (-1, 1)
  std::vector<double> g, w;
  g.reserve(grid);
  for (int i = 0; i < grid; ++i) {
    double x = -6.0 * sigma + (12.0 * sigma) * i / (grid - 1);
    if (i == grid - 1) x = 6.0 * sigma;
    if (density == TQ_DENS_BETA && !(std::fabs(x) < 1.0)) continue;
    g.push_back(x);
  }
  const int n = (int)g.size();
  if (n < 2 * K) return TQ_ERR_INVALID_ARG;
  w.resize(n);
  KSum tot;
  for (int i = 0; i < n; ++i) {
    w[i] = coord_density(g[i], d, density);
    tot.add(w[i]);
  }
  const double wsum = tot.value();
  for (int i = 0; i < n; ++i) w[i] /= wsum;
  // initial centroids: (k + 1/2)/K quantiles of the midpoint CDF, interpolated
  std::vector<double> cdf(n);
  {
    KSum run;
    for (int i = 0; i < n; ++i) {
      run.add(w[i]);
      cdf[i] = run.value() - 0.5 * w[i];
    }
  }
  std::vector<double> c(K), t(K - 1);
  for (int k = 0; k < K; ++k) {
    double q = (k + 0.5) / K;
    if (q <= cdf[0]) {
      c[k] = g[0];
      continue;
    }
    if (q >= cdf[n - 1]) {
      c[k] = g[n - 1];
      continue;
    }
    int i = (int)(std::upper_bound(cdf.begin(), cdf.end(), q) - cdf.begin()) - 1;
    c[k] = g[i] + (q - cdf[i]) * (g[i + 1] - g[i]) / (cdf[i + 1] - cdf[i]);
  }
  // Lloyd-Max ("TurboQuant 详解", section 痛点 2): thresholds at midpoints,
  // then each centroid moves to the weighted mean of its cell.
  std::vector<KSum> sw(K), swg(K);
  for (int it = 0; it < iters; ++it) {
    for (int k = 0; k + 1 < K; ++k) t[k] = 0.5 * (c[k] + c[k + 1]);
    for (int k = 0; k < K; ++k) sw[k] = KSum(), swg[k] = KSum();
    int cell = 0;
    for (int i = 0; i < n; ++i) {  // grid is ascending: the cell index only grows
      while (cell < K - 1 && g[i] >= t[cell]) ++cell;
      sw[cell].add(w[i]);
      swg[cell].add(w[i] * g[i]);
    }
    for (int k = 0; k < K; ++k) {
      double ws = sw[k].value();
      if (ws > 0.0) c[k] = swg[k].value() / ws;
    }
  }
  // symmetrise (the density is even)
  std::vector<double> cs(K);
  for (int k = 0; k < K; ++k) cs[k] = 0.5 * (c[k] - c[K - 1 - k]);
  for (int k = 0; k + 1 < K; ++k) t[k] = 0.5 * (cs[k] + cs[k + 1]);
  KSum dist;
  {
    int cell = 0;
    for (int i = 0; i < n; ++i) {
      while (cell < K - 1 && g[i] >= t[cell]) ++cell;
      double e = g[i] - cs[cell];
      dist.add(w[i] * e * e);
    }
  }
  std::memset(out, 0, sizeof(*out));
  out->d = d;
  out->b = b;
  out->density = density;
  out->grid = grid;
  out->iters = iters;
  const double sd = std::sqrt((double)d);
  for (int k = 0; k < K; ++k) out->centroid[k] = cs[k] * sd;
  for (int k = 0; k + 1 < K; ++k) out->threshold[k] = t[k] * sd;
  out->distortion = d * dist.value();
  return TQ_OK;
}

// ---------------------------------------------------------------- rotation
// Householder QR of G (row-major d×d); returns Π = Q·diag(sign(diag R)).
static tq_status haar_from_gaussian(int d, const double* G, double* Pi) {
  // column-major working copy: A[j*d + i] = G[i][j]
  std::vector<double> A((size_t)d * d), V((size_t)d * d, 0.0), vn(d, 0.0), rdiag(d, 0.0);
  for (int i = 0; i < d; ++i)
    for (int j = 0; j < d; ++j) A[(size_t)j * d + i] = G[(size_t)i * d + j];
  for (int k = 0; k < d; ++k) {
    double* col = &A[(size_t)k * d];
    KSum nrm;
    for (int i = k; i < d; ++i) nrm.add(col[i] * col[i]);
    double norm = std::sqrt(nrm.value());
    double alpha = col[k] > 0.0 ? -norm : norm;
    double* v = &V[(size_t)k * d];
    for (int i = k; i < d; ++i) v[i] = col[i];
    v[k] -= alpha;
    KSum vv;
    for (int i = k; i < d; ++i) vv.add(v[i] * v[i]);
    vn[k] = vv.value();
    rdiag[k] = alpha;
    if (vn[k] == 0.0) continue;
    const double inv = 2.0 / vn[k];
    parallel_for(d - k - 1, 64, [&](int a, int b) {
      for (int jj = a; jj < b; ++jj) {
        double* cj = &A[(size_t)(k + 1 + jj) * d];
        double dot = 0.0;
        for (int i = k; i < d; ++i) dot += v[i] * cj[i];
        dot *= inv;
        for (int i = k; i < d; ++i) cj[i] -= dot * v[i];
      }
    });
  }
  // Q = H_0 H_1 ... H_{d-1}, accumulated backwards into column-major Q
  std::vector<double> Q((size_t)d * d, 0.0);
  for (int i = 0; i < d; ++i) Q[(size_t)i * d + i] = 1.0;
  for (int k = d - 1; k >= 0; --k) {
    if (vn[k] == 0.0) continue;
    const double* v = &V[(size_t)k * d];
    const double inv = 2.0 / vn[k];
    parallel_for(d - k, 64, [&](int a, int b) {
      for (int jj = a; jj < b; ++jj) {
        double* qj = &Q[(size_t)(k + jj) * d];
        double dot = 0.0;
        for (int i = k; i < d; ++i) dot += v[i] * qj[i];
        dot *= inv;
        for (int i = k; i < d; ++i) qj[i] -= dot * v[i];
      }
    });
  }
  for (int i = 0; i < d; ++i)
    for (int j = 0; j < d; ++j) {
      double sgn = rdiag[j] < 0.0 ? -1.0 : 1.0;
      Pi[(size_t)i * d + j] = Q[(size_t)j * d + i] * sgn;
    }
  return TQ_OK;
}

// Hadamard matrix entry of order d = 2^k (Sylvester) or 12·2^k (Paley q = 11
// bordered matrix ⊗ Sylvester, row i = 2^k·a + j).
static int paley12(int a, int b) {
  if (a == b) return 1;  // H = I + S with S skew-symmetric, S_aa = 0
  if (a == 0) return 1;
  if (b == 0) return -1;
  static const int chi[11] = {0, 1, -1, 1, 1, 1, -1, -1, -1, 1, -1};  // residues 1,3,4,5,9
  return chi[((b - a) % 11 + 11) % 11];
}

static bool hadamard_order(int d, int* m_out, bool* paley) {
  if (d >= 1 && (d & (d - 1)) == 0) {
    *m_out = d;
    *paley = false;
    return true;
  }
  if (d % 12 == 0) {
    int m = d / 12;
    if (m >= 1 && (m & (m - 1)) == 0) {
      *m_out = m;
      *paley = true;
      return true;
    }
  }
  return false;
}

static int hadamard_entry(int d, int i, int j) {
  int m;
  bool pal;
  hadamard_order(d, &m, &pal);
  int s = (__builtin_popcount((unsigned)((i % m) & (j % m))) & 1) ? -1 : 1;
  if (pal) s *= paley12(i / m, j / m);
  return s;
}

// ---------------------------------------------------------------- fp16
static inline uint16_t h_bits(float f) {
  __half h = __float2half_rn(f);
  uint16_t u;
  std::memcpy(&u, &h, 2);
  return u;
}
static inline float h_val(uint16_t u) {
  __half h;
  std::memcpy(&h, &u, 2);
  return __half2float(h);
}
static inline uint32_t pack_h2(float lo, float hi) {
  return (uint32_t)h_bits(lo) | ((uint32_t)h_bits(hi) << 16);
}

static double pow2_near(double x) {  // power of two closest (in log) to x
  return std::ldexp(1.0, (int)std::lround(std::log2(x)));
}

// Encoder B fragments of the mma.m16n8k16 operand B[k][n] = scale·W[dim_out(n)][k]
// for chunk c of 128 output coordinates; n = 8j + 2t + e  <->  dim 128c + 32t + 2j + e.
// Stored per (chunk, kstep, ntile, plane, lane) as {b0, b1}.
static void encoder_fragments(const double* W, int d, double scale, std::vector<uint2>& out,
                              bool k_permuted) {
  const int chunks = (d + kChunk - 1) / kChunk;
  const int Kp = k_permuted ? kChunk : d;  // K extent
  const int KS = Kp / 16;
  out.assign((size_t)chunks * KS * 16 * 2 * 32, make_uint2(0, 0));
  auto dim_out = [&](int c, int n) {
    int j = n / 8, t = (n % 8) / 2, e = n % 2;
    return c * kChunk + 32 * t + 2 * j + e;
  };
  // input coordinate of K index kk: natural order for the rotation, and for the
  // QJL stage the order in which the rotation's accumulators are held:
  // kk = 16s + 8h + 2t + e  <->  dim 32t + 4s + 2h + e.
  auto dim_in = [&](int kk) {
    if (!k_permuted) return kk;
    int s = kk / 16, h = (kk % 16) / 8, t = (kk % 8) / 2, e = kk % 2;
    return 32 * t + 4 * s + 2 * h + e;
  };
  auto val = [&](int kk, int n, int c, int plane) -> float {
    int o = dim_out(c, n), i = dim_in(kk);
    if (o >= d || i >= d) return 0.f;
    double w = scale * W[(size_t)o * d + i];
    float hi = h_val(h_bits((float)w));
    if (plane == 0) return hi;
    return (float)(w - (double)hi);
  };
  for (int c = 0; c < chunks; ++c)
    for (int s = 0; s < KS; ++s)
      for (int j = 0; j < 16; ++j)
        for (int p = 0; p < 2; ++p)
          for (int lane = 0; lane < 32; ++lane) {
            int g = lane / 4, t = lane % 4;
            int n = 8 * j + g;
            int k0 = 16 * s + 2 * t, k1 = k0 + 8;
            uint2 f;
            f.x = pack_h2(val(k0, n, c, p), val(k0 + 1, n, c, p));
            f.y = pack_h2(val(k1, n, c, p), val(k1 + 1, n, c, p));
            out[((((size_t)c * KS + s) * 16 + j) * 2 + p) * 32 + lane] = f;
          }
}

// pi_scale·Π as the B operand of the tcgen05 encoder (d > 128): for output
// block ob (kUmmaTN coordinates), input chunk kc (kUmmaKC coordinates) and
// plane (0: fp16 of w, 1: fp16 of the remainder w - hi), one kUmmaTN x kUmmaKC
// tile in the no-swizzle K-major core-matrix order: 8 rows x 16 bytes per core
// matrix, 128 bytes between core matrices along K, 1024 bytes between 8-row
// groups.  Tile (ob, kc, plane) starts at ((ob·nkc + kc)·2 + plane)·kUmmaPlaneBytes.
static void umma_tiles(const double* W, int d, double scale, std::vector<uint16_t>& out) {
  const int nkc = d / kUmmaKC, nob = d / kUmmaTN;
  const size_t plane = kUmmaPlaneBytes / 2;
  out.assign((size_t)d * d * 2, 0);
  parallel_for(nob, 1, [&](int a, int bb) {
    for (int ob = a; ob < bb; ++ob)
      for (int kc = 0; kc < nkc; ++kc) {
        uint16_t* hi = out.data() + ((size_t)ob * nkc + kc) * 2 * plane;
        uint16_t* lo = hi + plane;
        for (int n = 0; n < kUmmaTN; ++n)
          for (int kk = 0; kk < kUmmaKC; ++kk) {
            const double w = scale * W[(size_t)(ob * kUmmaTN + n) * d + kc * kUmmaKC + kk];
            const uint16_t hb = h_bits((float)w);
            const size_t at = (size_t)(n / 8) * 512 + (kk / 8) * 64 + (n % 8) * 8 + (kk % 8);
            hi[at] = hb;
            lo[at] = h_bits((float)(w - (double)h_val(hb)));
          }
      }
  });
}

}  // namespace tq

using namespace tq;

// =========================================================================
extern "C" {

const char* tq_version(void) { return "tq 0.1 sm_103a"; }

const char* tq_status_string(tq_status s) {
  switch (s) {
    case TQ_OK: return "TQ_OK";
    case TQ_ERR_INVALID_ARG: return "TQ_ERR_INVALID_ARG";
    case TQ_ERR_UNSUPPORTED: return "TQ_ERR_UNSUPPORTED";
    case TQ_ERR_CUDA: return "TQ_ERR_CUDA";
    case TQ_ERR_ALLOC: return "TQ_ERR_ALLOC";
    case TQ_ERR_TIMEOUT: return "TQ_ERR_TIMEOUT";
  }
  return "TQ_ERR_UNKNOWN";
}

int tq_last_cuda_error(void) { return g_last_cuda_error.load(); }

tq_status tq_codebook_build(int d, int b, int density, int grid, int iters, tq_codebook* out) {
  if (!out || d < 2 || b < 1 || b > 4) return TQ_ERR_INVALID_ARG;
  if (density != TQ_DENS_BETA && density != TQ_DENS_GAUSS) return TQ_ERR_INVALID_ARG;
  if (grid <= 0) grid = 50000;
  if (iters <= 0) iters = 300;
  return build_codebook(d, b, density, grid, iters, out);
}

tq_status tq_rotation_haar(int d, const double* h_G, double* h_Pi) {
  if (d < 1 || d > kMaxD || !h_G || !h_Pi) return TQ_ERR_INVALID_ARG;
  try {
    return haar_from_gaussian(d, h_G, h_Pi);
  } catch (...) {
    return TQ_ERR_ALLOC;
  }
}

static bool d_supported(int d) {
  return d >= 32 && d <= kMaxD && d % 32 == 0 && (d <= kChunk || d % kChunk == 0);
}

tq_status tq_ctx_create(int d, int b, int mode, int rot_kind, const double* h_rot,
                        const double* h_S, const tq_codebook* cb, tq_ctx** out) {
  if (!out || !h_rot || !cb) return TQ_ERR_INVALID_ARG;
  *out = nullptr;
  if (mode != TQ_MSE && mode != TQ_PROD && mode != TQ_MIXED) return TQ_ERR_INVALID_ARG;
  if (rot_kind != TQ_ROT_DENSE && rot_kind != TQ_ROT_HADAMARD) return TQ_ERR_INVALID_ARG;
  if (b < 1 || b > 4 || (mode == TQ_PROD && b < 2) || (mode == TQ_MIXED && b > 3)) return TQ_ERR_INVALID_ARG;
  if (d % 32 != 0 || d < 32 || d > kMaxD) return TQ_ERR_INVALID_ARG;
  if (!d_supported(d)) return TQ_ERR_UNSUPPORTED;
  const int b_mse = mode == TQ_PROD ? b - 1 : b;
  if (cb->d != d || cb->b != b_mse) return TQ_ERR_INVALID_ARG;
  const bool mixed = mode == TQ_MIXED;
  if (mixed && (cb[1].d != d || cb[1].b != b + 1)) return TQ_ERR_INVALID_ARG;
  // b + 1/2 bits: the tensor-memory encoder, the scorer and decode at d = 128
  if (mixed && d != kChunk) return TQ_ERR_UNSUPPORTED;  // the d = 128 encoder, scorer and decode
  if (mode == TQ_PROD && !h_S) return TQ_ERR_INVALID_ARG;
  if (mode == TQ_PROD && d > kChunk) return TQ_ERR_UNSUPPORTED;
  int hm = 0;
  bool hp = false;
  if (rot_kind == TQ_ROT_HADAMARD && !hadamard_order(d, &hm, &hp)) return TQ_ERR_UNSUPPORTED;

  Ctx* c = new (std::nothrow) Ctx();
  if (!c) return TQ_ERR_ALLOC;
  c->cb = *cb;
  if (mixed) c->cb_hi = cb[1];
  const size_t dd = (size_t)d * d;
  c->h_pi = new (std::nothrow) double[dd];
  if (!c->h_pi) {
    delete c;
    return TQ_ERR_ALLOC;
  }
  if (rot_kind == TQ_ROT_DENSE) {
    std::memcpy(c->h_pi, h_rot, dd * sizeof(double));
  } else {
    const double inv = 1.0 / std::sqrt((double)d);
    for (int i = 0; i < d; ++i) {
      if (h_rot[i] != 1.0 && h_rot[i] != -1.0) {
        delete[] c->h_pi;
        delete c;
        return TQ_ERR_INVALID_ARG;
      }
    }
    for (int i = 0; i < d; ++i)
      for (int j = 0; j < d; ++j) c->h_pi[(size_t)i * d + j] = hadamard_entry(d, i, j) * h_rot[j] * inv;
  }
  if (mode == TQ_PROD) {
    c->h_s = new (std::nothrow) double[dd];
    if (!c->h_s) {
      delete[] c->h_pi;
      delete c;
      return TQ_ERR_ALLOC;
    }
    std::memcpy(c->h_s, h_S, dd * sizeof(double));
  }
  DevCtx& v = c->dev;
  std::memset(&v, 0, sizeof(v));
  v.d = d;
  v.b = b;
  v.b_mse = b_mse;
  v.mode = mode;
  v.rot = rot_kind;
  v.wait_limit = kWaitLimitDefault;
  v.words_per_vec = mixed ? mixed_words_per_vector(d, b) : words_per_vector(d, b_mse);
  v.qjl_words_per_vec = mode == TQ_PROD ? words_per_vector(d, 1) : 0;
  v.sqrt_d = (float)std::sqrt((double)d);
  v.pi_scale = (float)pow2_near(std::sqrt((double)d));
  const int K = 1 << b_mse;
  for (int k = 0; k < K; ++k) v.cen[k] = (float)cb->centroid[k];
  for (int k = 0; k + 1 < K; ++k) v.thr[k] = (float)cb->threshold[k];
  const int KH = mixed ? 2 * K : 0;  // TQ_MIXED: the (b+1)-bit codebook
  for (int k = 0; k < KH; ++k) v.cen_hi[k] = (float)cb[1].centroid[k];
  for (int k = 0; k + 1 < KH; ++k) v.thr_hi[k] = (float)cb[1].threshold[k];
  {
    auto symmetric = [](const float* thr, int n) {  // n thresholds, n odd
      const int h = n / 2;
      bool sym = thr[h] == 0.f;
      for (int j = 0; sym && j < h; ++j) sym = thr[h - 1 - j] == -thr[h + 1 + j];
      return sym;
    };
    v.sym_thr = symmetric(v.thr, K - 1) && (!mixed || symmetric(v.thr_hi, KH - 1)) ? 1 : 0;
  }
  if (mixed && !v.sym_thr) {  // only the tensor-memory encoder packs b + 1/2 bits
    delete[] c->h_pi;
    delete c;
    return TQ_ERR_UNSUPPORTED;
  }

  // alpha: scale that makes alpha·c_k closest to fp16 values (max relative
  // error); one alpha for both codebooks of TQ_MIXED, whose tables share the
  // logit and output scales
  {
    double best = 1e30, best_a = 1.0;
    for (int j = 0; j < 65536; ++j) {
      double a = 1.0 + j / 65536.0, worst = 0.0;
      for (int k = K / 2; k < K + KH; ++k) {
        double x = a * (k < K ? cb->centroid[k] : cb[1].centroid[k - K]);
        if (x == 0.0) continue;
        double r = std::fabs((double)h_val(h_bits((float)x)) - x) / std::fabs(x);
        worst = std::max(worst, r);
      }
      if (worst < best) {
        best = worst;
        best_a = a;
      }
    }
    v.alpha = (float)best_a;
  }

  // ---- device tables
  v.had_m = v.had_p = 0;
  if (rot_kind == TQ_ROT_HADAMARD) {
    v.had_m = hm;
    v.had_p = hp ? 12 : 1;
  }
  // d <= 128: mma.sync fragments; d > 128: tcgen05 tiles (unless the Hadamard
  // fast transform encodes without Π)
  const bool wht_path = rot_kind == TQ_ROT_HADAMARD && mode == TQ_MSE && v.had_m >= 32 && v.had_m <= 256;
  const bool umma_path = d > kChunk && d % kUmmaTN == 0 && mode == TQ_MSE && !wht_path;
  std::vector<uint2> frag_pi, frag_m;
  std::vector<uint16_t> umma, enc128, enc128m;
  if (d <= kChunk) encoder_fragments(c->h_pi, d, v.pi_scale, frag_pi, false);
  if (umma_path) umma_tiles(c->h_pi, d, v.pi_scale, umma);
  if (d == kChunk) umma_tiles(c->h_pi, d, v.pi_scale, enc128);  // the tcgen05 encoder at d = 128
  std::vector<double> M;
  if (mode == TQ_PROD) {
    M.assign(dd, 0.0);  // M = S·Πᵀ
    parallel_for(d, 8, [&](int a, int bb) {
      for (int j = a; j < bb; ++j)
        for (int i = 0; i < d; ++i) {
          double s = 0.0;
          for (int l = 0; l < d; ++l) s += c->h_s[(size_t)j * d + l] * c->h_pi[(size_t)i * d + l];
          M[(size_t)j * d + i] = s;
        }
    });
    double mx = 0.0;
    for (double x : M) mx = std::max(mx, std::fabs(x));
    v.m_scale = (float)pow2_near(4.0 / std::max(mx, 1e-30));
    encoder_fragments(M.data(), d, v.m_scale, frag_m, true);
    if (d == kChunk) umma_tiles(M.data(), d, v.m_scale, enc128m);
  }
  std::vector<float> pi32(dd), s32, slices, signs32;
  if (rot_kind == TQ_ROT_HADAMARD) {
    signs32.resize(d);
    for (int i = 0; i < d; ++i) signs32[i] = (float)h_rot[i];
  }
  for (size_t i = 0; i < dd; ++i) pi32[i] = (float)c->h_pi[i];
  if (d == kChunk) {  // Π in column slices for the decode rotation: [32-column slice][j][row][4]
    slices.resize(dd);
    for (int cc = 0; cc < d / 32; ++cc)
      for (int j = 0; j < 8; ++j)
        for (int r = 0; r < d; ++r)
          for (int e = 0; e < 4; ++e)
            slices[(((size_t)cc * 8 + j) * d + r) * 4 + e] = pi32[(size_t)r * d + 32 * cc + 4 * j + e];
  }
  std::vector<float> sslices;
  if (mode == TQ_PROD) {
    s32.resize(dd);
    for (size_t i = 0; i < dd; ++i) s32[i] = (float)c->h_s[i];
    if (d == kChunk) {  // S in the same column slices, for the query's S-rotation in decode
      sslices.resize(dd);
      for (int cc = 0; cc < d / 32; ++cc)
        for (int j = 0; j < 8; ++j)
          for (int r = 0; r < d; ++r)
            for (int e = 0; e < 4; ++e)
              sslices[(((size_t)cc * 8 + j) * d + r) * 4 + e] = s32[(size_t)r * d + 32 * cc + 4 * j + e];
    }
  }
  const int E = 1 << (2 * b_mse);
  std::vector<uint32_t> lut(E);
  for (int p = 0; p < E; ++p) {
    int k0 = p & (K - 1), k1 = p >> b_mse;
    lut[p] = pack_h2((float)(v.alpha * cb->centroid[k0]), (float)(v.alpha * cb->centroid[k1]));
  }
  std::vector<uint32_t> lut_hi(mixed ? (size_t)1 << (2 * (b + 1)) : 0);
  for (size_t p = 0; p < lut_hi.size(); ++p) {
    const int k0 = (int)(p & (size_t)(KH - 1)), k1 = (int)(p >> (b + 1));
    lut_hi[p] = pack_h2((float)(v.alpha * cb[1].centroid[k0]), (float)(v.alpha * cb[1].centroid[k1]));
  }

  auto al = [](size_t x) { return (x + 255) / 256 * 256; };
  size_t o_pi = 0;
  size_t o_m = o_pi + al(frag_pi.size() * sizeof(uint2));
  size_t o_p32 = o_m + al(frag_m.size() * sizeof(uint2));
  size_t o_s32 = o_p32 + al(pi32.size() * sizeof(float));
  size_t o_sl = o_s32 + al(s32.size() * sizeof(float));
  size_t o_sg = o_sl + al(slices.size() * sizeof(float));
  size_t o_ss = o_sg + al(signs32.size() * sizeof(float));
  size_t o_um = o_ss + al(sslices.size() * sizeof(float));
  size_t o_e1 = o_um + al(umma.size() * sizeof(uint16_t));
  size_t o_e2 = o_e1 + al(enc128.size() * sizeof(uint16_t));
  size_t o_lut = o_e2 + al(enc128m.size() * sizeof(uint16_t));
  size_t o_lh = o_lut + al(lut.size() * sizeof(uint32_t));
  size_t o_st = o_lh + al(lut_hi.size() * sizeof(uint32_t));
  size_t total = o_st + 256;
  void* dmem = nullptr;
  cudaError_t e = cudaMalloc(&dmem, total);
  if (e != cudaSuccess) {
    delete[] c->h_pi;
    delete[] c->h_s;
    delete c;
    (void)cudaGetLastError();
    return TQ_ERR_ALLOC;
  }
  char* base = (char*)dmem;
  auto up = [&](size_t off, const void* src, size_t n) -> cudaError_t {
    if (n == 0) return cudaSuccess;
    return cudaMemcpy(base + off, src, n, cudaMemcpyHostToDevice);
  };
  e = up(o_pi, frag_pi.data(), frag_pi.size() * sizeof(uint2));
  if (e == cudaSuccess) e = up(o_m, frag_m.data(), frag_m.size() * sizeof(uint2));
  if (e == cudaSuccess) e = up(o_p32, pi32.data(), pi32.size() * sizeof(float));
  if (e == cudaSuccess) e = up(o_s32, s32.data(), s32.size() * sizeof(float));
  if (e == cudaSuccess) e = up(o_sl, slices.data(), slices.size() * sizeof(float));
  if (e == cudaSuccess) e = up(o_sg, signs32.data(), signs32.size() * sizeof(float));
  if (e == cudaSuccess) e = up(o_ss, sslices.data(), sslices.size() * sizeof(float));
  if (e == cudaSuccess) e = up(o_um, umma.data(), umma.size() * sizeof(uint16_t));
  if (e == cudaSuccess) e = up(o_e1, enc128.data(), enc128.size() * sizeof(uint16_t));
  if (e == cudaSuccess) e = up(o_e2, enc128m.data(), enc128m.size() * sizeof(uint16_t));
  if (e == cudaSuccess) e = up(o_lut, lut.data(), lut.size() * sizeof(uint32_t));
  if (e == cudaSuccess) e = up(o_lh, lut_hi.data(), lut_hi.size() * sizeof(uint32_t));
  if (e == cudaSuccess) e = cudaMemset(base + o_st, 0, 256);
  if (e != cudaSuccess) {
    cudaFree(dmem);
    delete[] c->h_pi;
    delete[] c->h_s;
    delete c;
    return set_cuda_error(e);
  }
  c->d_alloc = dmem;
  c->d_bytes = total;
  v.enc_pi = d <= kChunk ? (const uint2*)(base + o_pi) : nullptr;
  v.umma_tab = umma_path ? (const unsigned char*)(base + o_um) : nullptr;
  v.enc_tab = enc128.empty() ? nullptr : (const unsigned char*)(base + o_e1);
  v.enc_tab_m = enc128m.empty() ? nullptr : (const unsigned char*)(base + o_e2);
  v.s_slices = sslices.empty() ? nullptr : (const float4*)(base + o_ss);
  v.enc_m = mode == TQ_PROD ? (const uint2*)(base + o_m) : nullptr;
  v.pi = (const float*)(base + o_p32);
  v.s_mat = mode == TQ_PROD ? (const float*)(base + o_s32) : nullptr;
  v.pi_slices = d == kChunk ? (const float4*)(base + o_sl) : nullptr;
  v.signs = rot_kind == TQ_ROT_HADAMARD ? (const float*)(base + o_sg) : nullptr;
  v.lut = (const uint32_t*)(base + o_lut);
  v.lut_hi = mixed ? (const uint32_t*)(base + o_lh) : nullptr;
  v.status = (int*)(base + o_st);
  // the fast transform's one-time launch setup now, outside any stream capture
  // (its launches then depend on nothing done before them; a failure here
  // shows again, and is reported, at the first encode)
  if (d != kChunk) (void)prime_encode_wht(v);
  *out = reinterpret_cast<tq_ctx*>(c);
  return TQ_OK;
}

tq_status tq_ctx_set_wait_limit(tq_ctx* ctx, uint32_t polls) {
  if (!ctx) return TQ_ERR_INVALID_ARG;
  reinterpret_cast<Ctx*>(ctx)->dev.wait_limit = polls;
  return TQ_OK;
}

tq_status tq_ctx_destroy(tq_ctx* ctx) {
  if (!ctx) return TQ_ERR_INVALID_ARG;
  Ctx* c = reinterpret_cast<Ctx*>(ctx);
  cudaError_t e = cudaSuccess;
  if (c->d_alloc) e = cudaFree(c->d_alloc);
  delete[] c->h_pi;
  delete[] c->h_s;
  delete c;
  return e == cudaSuccess ? TQ_OK : set_cuda_error(e);
}

tq_status tq_codes_layout(const tq_ctx* ctx, int layout, int64_t n, tq_codes* desc,
                          size_t* codes_bytes, size_t* norm_bytes, size_t* qjl_bytes,
                          size_t* rnorm_bytes) {
  if (!ctx || !desc || n < 0) return TQ_ERR_INVALID_ARG;
  if (layout != TQ_LAYOUT_TOKEN && layout != TQ_LAYOUT_PAIR) return TQ_ERR_INVALID_ARG;
  const DevCtx& v = reinterpret_cast<const Ctx*>(ctx)->dev;
  std::memset(desc, 0, sizeof(*desc));
  desc->n = n;
  desc->d = v.d;
  desc->b_mse = v.b_mse;
  desc->mode = v.mode;
  desc->layout = layout;
  desc->words_per_vec = v.words_per_vec;
  desc->qjl_words_per_vec = v.qjl_words_per_vec;
  int64_t nn = layout == TQ_LAYOUT_PAIR ? (n + 1) / 2 * 2 : n;
  if (codes_bytes) *codes_bytes = (size_t)nn * v.words_per_vec * 4;
  if (norm_bytes) *norm_bytes = (size_t)n * 4;
  if (qjl_bytes) *qjl_bytes = (size_t)n * v.qjl_words_per_vec * 4;
  if (rnorm_bytes) *rnorm_bytes = v.mode == TQ_PROD ? (size_t)n * 4 : 0;
  return TQ_OK;
}

static bool al16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

static tq_status check_codes(const DevCtx& v, const tq_codes* c) {
  if (!c || !c->d_codes || !c->d_norm || c->n < 0) return TQ_ERR_INVALID_ARG;
  if (c->d != v.d || c->b_mse != v.b_mse || c->mode != v.mode) return TQ_ERR_INVALID_ARG;
  if (c->words_per_vec != v.words_per_vec) return TQ_ERR_INVALID_ARG;
  if (c->layout != TQ_LAYOUT_TOKEN && c->layout != TQ_LAYOUT_PAIR) return TQ_ERR_INVALID_ARG;
  if (!al16(c->d_codes)) return TQ_ERR_INVALID_ARG;
  if (v.mode == TQ_PROD) {
    if (!c->d_qjl || !c->d_rnorm || c->qjl_words_per_vec != v.qjl_words_per_vec || !al16(c->d_qjl))
      return TQ_ERR_INVALID_ARG;
  }
  return TQ_OK;
}

tq_status tq_encode(const tq_ctx* ctx, const void* d_x, int x_dtype, int64_t N,
                    const tq_codes* out, int64_t offset, int64_t group_rows, int64_t group_stride,
                    tq_stream stream) {
  if (!ctx || !out) return TQ_ERR_INVALID_ARG;
  const DevCtx& v = reinterpret_cast<const Ctx*>(ctx)->dev;
  if (x_dtype != TQ_F32 && x_dtype != TQ_F16) return TQ_ERR_INVALID_ARG;
  if (N < 0 || offset < 0 || group_rows <= 0 || group_stride < 0) return TQ_ERR_INVALID_ARG;
  tq_status st = check_codes(v, out);
  if (st != TQ_OK) return st;
  if (N == 0) return TQ_OK;
  if (!d_x || !al16(d_x)) return TQ_ERR_INVALID_ARG;
  // d = 128 takes the tensor-memory encoder for every rotation: the product
  // with the materialized H·D/√d costs it nothing (its epilogue bounds it),
  // and it ran faster than the butterflies of the fast transform
  const bool wht = wht_supported(v) && out->layout == TQ_LAYOUT_TOKEN && !enc128_supported(v);
  const bool wide = !wht && v.d > kChunk;
  if (wide && (!umma_supported(v) || out->layout != TQ_LAYOUT_TOKEN)) return TQ_ERR_UNSUPPORTED;
  // every destination index must lie inside the code set
  int64_t groups = (N + group_rows - 1) / group_rows;
  int64_t last_in_group = std::min<int64_t>(group_rows, N) - 1;
  int64_t max_dst = (groups - 1) * group_stride + offset + last_in_group;
  if (max_dst >= out->n) return TQ_ERR_INVALID_ARG;
  if (groups > 1 && group_stride < group_rows) return TQ_ERR_INVALID_ARG;  // no overlap
  if (wht)
    return launch_encode_wht(v, d_x, x_dtype, N, out, offset, group_rows, group_stride, (cudaStream_t)stream);
  if (wide)
    return launch_encode_umma(v, d_x, x_dtype, N, out, offset, group_rows, group_stride, (cudaStream_t)stream);
  if (enc128_supported(v))
    return launch_encode128(v, d_x, x_dtype, N, out, offset, group_rows, group_stride, (cudaStream_t)stream);
  return launch_encode(v, d_x, x_dtype, N, out, offset, group_rows, group_stride,
                       (cudaStream_t)stream);
}

tq_status tq_scores_workspace_size(const tq_ctx* ctx, int M, size_t* bytes) {
  if (!ctx || !bytes || M < 0) return TQ_ERR_INVALID_ARG;
  *bytes = scores_ws_bytes(reinterpret_cast<const Ctx*>(ctx)->dev, M);
  return TQ_OK;
}

tq_status tq_scores(const tq_ctx* ctx, const float* d_q, int M, const tq_codes* keys,
                    int64_t first, int64_t N, float* d_scores, void* d_ws, size_t ws_bytes,
                    tq_stream stream) {
  if (!ctx || !keys) return TQ_ERR_INVALID_ARG;
  const DevCtx& v = reinterpret_cast<const Ctx*>(ctx)->dev;
  tq_status st = check_codes(v, keys);
  if (st != TQ_OK) return st;
  if (keys->layout != TQ_LAYOUT_TOKEN) return TQ_ERR_INVALID_ARG;
  if (M < 0 || N < 0 || first < 0 || first + N > keys->n) return TQ_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return TQ_OK;
  if (!d_q || !d_scores || !d_ws || !al16(d_ws) || !al16(d_q)) return TQ_ERR_INVALID_ARG;
  if (ws_bytes < scores_ws_bytes(v, M)) return TQ_ERR_INVALID_ARG;
  if (v.d != kChunk) return TQ_ERR_UNSUPPORTED;
  return launch_scores(v, d_q, M, keys, first, N, d_scores, d_ws, ws_bytes, (cudaStream_t)stream);
}

tq_status tq_decode_workspace_size(const tq_ctx* kctx, int B, int Hq, int Hkv, int64_t seq,
                                   size_t* bytes) {
  if (!kctx || !bytes || B < 0 || Hq < 0 || Hkv <= 0 || seq < 0) return TQ_ERR_INVALID_ARG;
  *bytes = decode_ws_bytes(reinterpret_cast<const Ctx*>(kctx)->dev.d, B, Hq, Hkv, seq);
  return TQ_OK;
}

tq_status tq_decode_attention(const tq_ctx* kctx, const tq_ctx* vctx, const void* d_q,
                              int q_dtype, const tq_codes* K, const tq_codes* V, int B, int Hq,
                              int Hkv, int64_t seq, int64_t cap, float scale, float* d_out,
                              void* d_ws, size_t ws_bytes, tq_stream stream) {
  if (!kctx || !vctx || !K || !V) return TQ_ERR_INVALID_ARG;
  const DevCtx& kc = reinterpret_cast<const Ctx*>(kctx)->dev;
  const DevCtx& vc = reinterpret_cast<const Ctx*>(vctx)->dev;
  if ((vc.mode != TQ_MSE && vc.mode != TQ_MIXED) || kc.d != vc.d) return TQ_ERR_INVALID_ARG;  // values MSE or b + 1/2 bits
  tq_status st = check_codes(kc, K);
  if (st != TQ_OK) return st;
  st = check_codes(vc, V);
  if (st != TQ_OK) return st;
  if (K->layout != TQ_LAYOUT_TOKEN || V->layout != TQ_LAYOUT_PAIR) return TQ_ERR_INVALID_ARG;
  if (q_dtype != TQ_F32 && q_dtype != TQ_F16) return TQ_ERR_INVALID_ARG;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || seq <= 0 || cap < seq || (cap & 1))
    return TQ_ERR_INVALID_ARG;
  const int gqa = Hq / Hkv;
  if (gqa != 1 && gqa != 2 && gqa != 4 && gqa != 8) return TQ_ERR_UNSUPPORTED;
  if ((int64_t)B * Hkv * cap > K->n || (int64_t)B * Hkv * cap > V->n) return TQ_ERR_INVALID_ARG;
  if (!d_q || !d_out || !d_ws || !al16(d_ws) || !al16(d_q)) return TQ_ERR_INVALID_ARG;
  if (!al16(K->d_norm) || !al16(V->d_norm)) return TQ_ERR_INVALID_ARG;
  if (ws_bytes < decode_ws_bytes(kc.d, B, Hq, Hkv, seq)) return TQ_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return TQ_ERR_INVALID_ARG;
  if (kc.d != kChunk) return TQ_ERR_UNSUPPORTED;
  return launch_decode(kc, vc, d_q, q_dtype, K, V, B, Hq, Hkv, seq, cap, scale, d_out, d_ws,
                       ws_bytes, (cudaStream_t)stream);
}

tq_status tq_decode_step(const tq_ctx* kctx, const tq_ctx* vctx, const void* d_q, int q_dtype,
                         const void* d_k_new, const void* d_v_new, int new_dtype, const tq_codes* K,
                         const tq_codes* V, int B, int Hq, int Hkv, int64_t seq, int64_t cap,
                         float scale, float* d_out, void* d_ws, size_t ws_bytes,
                         tq_stream stream) {
  if (!kctx || !vctx || !K || !V) return TQ_ERR_INVALID_ARG;
  const DevCtx& kc = reinterpret_cast<const Ctx*>(kctx)->dev;
  const DevCtx& vc = reinterpret_cast<const Ctx*>(vctx)->dev;
  if ((vc.mode != TQ_MSE && vc.mode != TQ_MIXED) || kc.d != vc.d) return TQ_ERR_INVALID_ARG;
  if (kc.mode != TQ_MSE) return TQ_ERR_UNSUPPORTED;  // the fused append encodes MSE keys only
  tq_status st = check_codes(kc, K);
  if (st != TQ_OK) return st;
  st = check_codes(vc, V);
  if (st != TQ_OK) return st;
  if (K->layout != TQ_LAYOUT_TOKEN || V->layout != TQ_LAYOUT_PAIR) return TQ_ERR_INVALID_ARG;
  if (q_dtype != TQ_F32 && q_dtype != TQ_F16) return TQ_ERR_INVALID_ARG;
  if (new_dtype != TQ_F32 && new_dtype != TQ_F16) return TQ_ERR_INVALID_ARG;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || seq <= 0 || cap < seq || (cap & 1))
    return TQ_ERR_INVALID_ARG;
  const int gqa = Hq / Hkv;
  if (gqa != 1 && gqa != 2 && gqa != 4 && gqa != 8) return TQ_ERR_UNSUPPORTED;
  if ((int64_t)B * Hkv * cap > K->n || (int64_t)B * Hkv * cap > V->n) return TQ_ERR_INVALID_ARG;
  if (!d_q || !d_out || !d_k_new || !d_v_new || !al16(d_q) || !al16(d_k_new) || !al16(d_v_new))
    return TQ_ERR_INVALID_ARG;
  if (!d_ws || !al16(d_ws) || ws_bytes < decode_ws_bytes(kc.d, B, Hq, Hkv, seq))
    return TQ_ERR_INVALID_ARG;
  if (!al16(K->d_norm) || !al16(V->d_norm)) return TQ_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return TQ_ERR_INVALID_ARG;
  if (kc.d != kChunk) return TQ_ERR_UNSUPPORTED;
  return launch_step(kc, vc, d_q, q_dtype, d_k_new, d_v_new, new_dtype, K, V, B, Hq, Hkv, seq, cap,
                     scale, d_out, d_ws, (cudaStream_t)stream);
}

// Same checks as tq_decode_attention, without the workspace arguments.
tq_status tq_decode_attention_noalloc(const tq_ctx* kctx, const tq_ctx* vctx, const void* d_q,
                                      int q_dtype, const tq_codes* K, const tq_codes* V, int B,
                                      int Hq, int Hkv, int64_t seq, int64_t cap, float scale,
                                      float* d_out, tq_stream stream) {
  if (!kctx || !vctx || !K || !V) return TQ_ERR_INVALID_ARG;
  const DevCtx& kc = reinterpret_cast<const Ctx*>(kctx)->dev;
  const DevCtx& vc = reinterpret_cast<const Ctx*>(vctx)->dev;
  if ((vc.mode != TQ_MSE && vc.mode != TQ_MIXED) || kc.d != vc.d) return TQ_ERR_INVALID_ARG;  // values MSE or b + 1/2 bits
  tq_status st = check_codes(kc, K);
  if (st != TQ_OK) return st;
  st = check_codes(vc, V);
  if (st != TQ_OK) return st;
  if (K->layout != TQ_LAYOUT_TOKEN || V->layout != TQ_LAYOUT_PAIR) return TQ_ERR_INVALID_ARG;
  if (q_dtype != TQ_F32 && q_dtype != TQ_F16) return TQ_ERR_INVALID_ARG;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || seq <= 0 || cap < seq || (cap & 1))
    return TQ_ERR_INVALID_ARG;
  const int gqa = Hq / Hkv;
  if (gqa != 1 && gqa != 2 && gqa != 4 && gqa != 8) return TQ_ERR_UNSUPPORTED;
  if (decode_ws_bytes(kc.d, B, Hq, Hkv, seq) > decode_noalloc_limit()) return TQ_ERR_UNSUPPORTED;
  if ((int64_t)B * Hkv * cap > K->n || (int64_t)B * Hkv * cap > V->n) return TQ_ERR_INVALID_ARG;
  if (!d_q || !d_out || !al16(d_q)) return TQ_ERR_INVALID_ARG;
  if (!al16(K->d_norm) || !al16(V->d_norm)) return TQ_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return TQ_ERR_INVALID_ARG;
  if (kc.d != kChunk) return TQ_ERR_UNSUPPORTED;
  return launch_decode_noalloc(kc, vc, d_q, q_dtype, K, V, B, Hq, Hkv, seq, cap, scale, d_out,
                               (cudaStream_t)stream);
}

tq_status tq_unpack_indices(const tq_codes* codes, int64_t first, int64_t count, uint8_t* h_idx,
                            uint8_t* h_bits) {
  if (!codes || !codes->d_codes || !h_idx || first < 0 || count < 0 || first + count > codes->n)
    return TQ_ERR_INVALID_ARG;
  if (count == 0) return TQ_OK;
  const int d = codes->d, b = codes->b_mse, W = codes->words_per_vec;
  const bool pair = codes->layout == TQ_LAYOUT_PAIR, mixed = codes->mode == TQ_MIXED;
  // copy the covering range of words
  int64_t v0 = pair ? first / 2 * 2 : first;
  int64_t v1 = pair ? (first + count + 1) / 2 * 2 : first + count;
  std::vector<uint32_t> w((size_t)(v1 - v0) * W);
  cudaError_t e = cudaMemcpy(w.data(), codes->d_codes + (size_t)v0 * W, w.size() * 4,
                             cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return set_cuda_error(e);
  for (int64_t r = 0; r < count; ++r) {
    int64_t vi = first + r;
    for (int j = 0; j < d; ++j) {
      int64_t bitpos;
      const uint32_t* base;
      const int wj = mixed ? mixed_width(j, b) : b;
      const int64_t pj = mixed ? mixed_pos(j, b) : (int64_t)j * b;
      if (!pair) {
        base = &w[(size_t)(vi - v0) * W];
        bitpos = pj;
      } else {
        base = &w[(size_t)(vi / 2 * 2 - v0) * W];
        bitpos = 2 * pj + (vi & 1) * wj;
      }
      int code = 0;
      for (int k = 0; k < wj; ++k) {
        int64_t p = bitpos + k;
        code |= ((base[p / 32] >> (p % 32)) & 1u) << k;
      }
      h_idx[r * d + j] = (uint8_t)code;
    }
  }
  if (h_bits) {
    if (codes->mode != TQ_PROD || !codes->d_qjl) return TQ_ERR_INVALID_ARG;
    const int QW = codes->qjl_words_per_vec;
    std::vector<uint32_t> q((size_t)count * QW);
    e = cudaMemcpy(q.data(), codes->d_qjl + (size_t)first * QW, q.size() * 4,
                   cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return set_cuda_error(e);
    for (int64_t r = 0; r < count; ++r)
      for (int j = 0; j < d; ++j) h_bits[r * d + j] = (uint8_t)((q[r * QW + j / 32] >> (j % 32)) & 1u);
  }
  return TQ_OK;
}

tq_status tq_status_poll(const tq_ctx* ctx, tq_stream stream) {
  if (!ctx) return TQ_ERR_INVALID_ARG;
  const DevCtx& v = reinterpret_cast<const Ctx*>(ctx)->dev;
  int h = 0;
  cudaError_t e = cudaMemcpyAsync(&h, v.status, sizeof(int), cudaMemcpyDeviceToHost,
                                  (cudaStream_t)stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e == cudaSuccess && h != 0) e = cudaMemsetAsync(v.status, 0, sizeof(int), (cudaStream_t)stream);
  if (e != cudaSuccess) return set_cuda_error(e);
  return h == 0 ? TQ_OK : TQ_ERR_TIMEOUT;
}

}  // extern "C"
