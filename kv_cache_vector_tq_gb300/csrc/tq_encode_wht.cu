// TurboQuant_MSE encoder with the randomized Hadamard rotation, as a fast
// transform instead of a dense d x d product.
//
// "压缩与速度的博弈——TurboQuant 和 RotorQuant 的真相" (the WHT-based rotation):
// Π = H·diag(σ)/√d with H a Hadamard matrix and σ random signs.  For
// d = P·m (P = 1, or P = 12 with H = H12 ⊗ H_m, H12 the Paley matrix of
// order 12 and H_m Sylvester of order m = 2^k):
//   z = H·(σ ∘ x),  y = z/√d,  and the unit-variance coordinate is
//   v = √d·y/‖x‖ = z/‖x‖,
// so the transform needs only additions and subtractions of the input.
// Per vector ("TurboQuant 详解", section 一个具体例子 steps 1-6): s = ‖x‖,
// idx_i = #{k : v_i >= t_k}, pack, store s.
//
// Work split: one warp per Hadamard block of a vector (the twelve blocks of a
// d = 12·m vector are the twelve warps of a CTA; for d = m, eight vectors per
// CTA), lane L holding elements 32k + L of its block.  Rows stream into a
// three-slot shared-memory ring by cp.async, two row groups ahead of the one
// being transformed; the grid holds as many CTAs as are resident at once.
// Plain fp32 butterflies: each output sees one rounding per stage, so the
// error in v stays near √(log2 d)·2^-24 (about 2e-7 at d = 3072), inside the
// 1e-6 band around the codebook thresholds.
#include <algorithm>

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {

struct WhtParams {
  const void* x;
  int64_t N;
  int d, m;
  uint32_t* codes;
  float* norm;
  int W;
  const float* signs;  // σ, d entries of ±1
  float thr[15];
  int sym;             // thresholds symmetric about 0
  int64_t offset, group_rows, group_stride;
};

// Paley Hadamard matrix of order 12 (the q = 11 construction, H = I + S with S
// skew-symmetric): the same entries as the host table the dense path uses.
__host__ __device__ constexpr int paley12_sign(int a, int b) {
  // residues mod 11: 1, 3, 4, 5, 9
  return a == b ? 1
         : a == 0 ? 1
         : b == 0 ? -1
         : ((((b - a) % 11 + 11) % 11) == 1 || (((b - a) % 11 + 11) % 11) == 3 ||
            (((b - a) % 11 + 11) % 11) == 4 || (((b - a) % 11 + 11) % 11) == 5 ||
            (((b - a) % 11 + 11) % 11) == 9)
             ? 1
             : -1;
}

// The kernel's circulant form of rows 1-11: the +1 entries off the diagonal
// of row a >= 1 sit at b = (a + o) % 11 + 1 for o in {0, 2, 3, 4, 8}.
__host__ __device__ constexpr bool paley12_residue_form() {
  for (int a = 1; a < 12; ++a)
    for (int b = 1; b < 12; ++b) {
      if (b == a) continue;
      const bool listed = b == (a + 0) % 11 + 1 || b == (a + 2) % 11 + 1 || b == (a + 3) % 11 + 1 ||
                          b == (a + 4) % 11 + 1 || b == (a + 8) % 11 + 1;
      if (listed != (paley12_sign(a, b) > 0)) return false;
    }
  for (int a = 1; a < 12; ++a)
    if (paley12_sign(a, 0) != -1 || paley12_sign(a, a) != 1 || paley12_sign(0, a) != 1) return false;
  return paley12_sign(0, 0) == 1;
}
static_assert(paley12_residue_form(), "circulant form of the Paley matrix");

constexpr int kWhtStages = 3;  // row groups in flight per CTA (cp.async ring)

__device__ __forceinline__ void wcp16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void wcp_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
// Code of v: #{k : v >= t_k}, branch-free with the thresholds in registers
// (kernel parameters): the sign bit of each difference counts a threshold
// above v.  Symmetric codebooks compare |v| with the positive half only.
template <int BM>
__device__ __forceinline__ int wht_code(float v, const float (&thr)[15], bool sym) {
  constexpr int H = (1 << (BM - 1)) - 1;
  constexpr uint32_t kAll = (1u << BM) - 1u;
  uint32_t above = 0u;
  if (sym) {
    const float a = fabsf(v);
#pragma unroll
    for (int j = 0; j < H; ++j) above += __float_as_uint(a - thr[H + 1 + j]) >> 31;
    // v >= 0 (-0 included, as the search it replaces): kAll - above; v < 0: above
    return (int)(v >= 0.f ? kAll - above : above);
  }
#pragma unroll
  for (int k = 0; k < 2 * H + 1; ++k) above += __float_as_uint(v - thr[k]) >> 31;
  return (int)(kAll - above);
}

template <int N>
__device__ __forceinline__ void wcp_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// Pack the vector's codes (one byte per coordinate in `cb`) into word w of
// the canonical stream: code j at bits [j·BM, j·BM + BM).
template <int BM>
__device__ __forceinline__ uint32_t pack_word(const unsigned char* cb, int w, int d) {
  if constexpr (BM == 4) {  // eight codes: two 4-byte reads, bytes folded into nibbles
    const uint2 u = *reinterpret_cast<const uint2*>(cb + 8 * w);
    uint32_t lo = (u.x | (u.x >> 4)) & 0x00FF00FFu, hi = (u.y | (u.y >> 4)) & 0x00FF00FFu;
    lo = (lo | (lo >> 8)) & 0xFFFFu;
    hi = (hi | (hi >> 8)) & 0xFFFFu;
    return lo | (hi << 16);
  } else {
    uint32_t word = 0u;
    const int c0 = (32 * w) / BM, c1 = min(d, (32 * w + 32 + BM - 1) / BM);
    for (int c = c0; c < c1; ++c) {
      const int sh = c * BM - 32 * w;  // negative for a code straddling into this word
      const uint32_t code = cb[c];
      word |= sh >= 0 ? code << sh : code >> (-sh);
    }
    return word;
  }
}

// Warp w of a CTA owns block a of one vector: P = 12 -> the CTA is one vector
// (12 warps, a = w); P = 1 -> eight vectors, one warp each.  Lane L holds the
// E = m/32 elements i' = 32k + L of its block, so the Sylvester stages with
// h >= 32 run in registers and those with h < 32 by warp shuffles; the Paley
// stage (P = 12) is the one exchange through shared memory.
template <int BM, int P, int E, bool F16>
__global__ void __launch_bounds__(P == 12 ? 384 : 256) encode_wht_kernel(const WhtParams p) {
  constexpr int NW = P == 12 ? 12 : 8;  // warps per CTA
  constexpr int VPC = P == 12 ? 1 : 8;  // vectors per CTA
  constexpr int M = 32 * E;             // Sylvester order
  constexpr int D = P * M;
  constexpr int ES = F16 ? 2 : 4;
  constexpr int SLOT = VPC * D * ES;    // a ring slot: the CTA's VPC consecutive rows
  extern __shared__ __align__(16) unsigned char wsm[];
  float* zs = reinterpret_cast<float*>(wsm);                    // [D] Paley exchange (P = 12)
  float* part = zs + (P == 12 ? D : 0);                        // [12] warp norm partials, [16 + 12] rescaled ones
  unsigned char* cbuf = reinterpret_cast<unsigned char*>(part + 32);  // [VPC][D] code bytes
  unsigned char* ring = cbuf + ((VPC * D + 15) / 16) * 16;
  __shared__ float thr_s[16];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int vloc = P == 12 ? 0 : warp, a = P == 12 ? warp : 0;
  if (tid < 16) thr_s[tid] = tid < (1 << BM) - 1 ? p.thr[tid] : INFINITY;
  float sg[E];
#pragma unroll
  for (int k = 0; k < E; ++k) sg[k] = p.signs[a * M + 32 * k + lane];
  const int64_t stride_rows = (int64_t)gridDim.x * VPC;
  auto fetch = [&](int64_t first_row, int slot) {
    unsigned char* dst = ring + slot * SLOT;
    const int64_t avail = min((int64_t)VPC, p.N - first_row);
    for (int i = tid; i < SLOT / 16; i += NW * 32) {
      if (i / (D * ES / 16) < avail)
        wcp16(dst + i * 16, static_cast<const unsigned char*>(p.x) + first_row * D * ES + (int64_t)i * 16);
      else
        *reinterpret_cast<uint4*>(dst + i * 16) = make_uint4(0u, 0u, 0u, 0u);
    }
    wcp_commit();
  };
#pragma unroll
  for (int k = 0; k < kWhtStages - 1; ++k) fetch((int64_t)blockIdx.x * VPC + k * stride_rows, k);
  __syncthreads();

  int it = 0;
  for (int64_t base = (int64_t)blockIdx.x * VPC; base < p.N; base += stride_rows, ++it) {
    // the slot refilled now was read last iteration; with P = 1 the warps do
    // not meet after that read, so they do here
    if constexpr (P == 1) __syncthreads();
    fetch(base + (kWhtStages - 1) * stride_rows, (it + kWhtStages - 1) % kWhtStages);
    wcp_wait<kWhtStages - 1>();
    __syncthreads();  // this group's rows are in; the previous group's buffers are free
    const unsigned char* src = ring + (it % kWhtStages) * SLOT + vloc * D * ES;
    float x[E];
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < E; ++k) {
      const int o = a * M + 32 * k + lane;
      x[k] = F16 ? __half2float(reinterpret_cast<const __half*>(src)[o]) : reinterpret_cast<const float*>(src)[o];
      ss = fmaf(x[k], x[k], ss);
      x[k] *= sg[k];
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(kFull, ss, off);
    // Sylvester stages of order M over i' = 32k + L
#pragma unroll
    for (int hk = 1; hk < E; hk <<= 1)  // h = 32·hk: partners k and k ^ hk, in registers
#pragma unroll
      for (int k = 0; k < E; ++k)
        if (!(k & hk)) {
          const float u = x[k], v = x[k | hk];
          x[k] = u + v;
          x[k | hk] = u - v;
        }
#pragma unroll
    for (int h = 1; h < 32; h <<= 1) {  // h < 32: partner lane L ^ h
      const float sgn = (lane & h) ? -1.f : 1.f;
#pragma unroll
      for (int k = 0; k < E; ++k) x[k] = fmaf(sgn, x[k], __shfl_xor_sync(kFull, x[k], h));
    }
    // squares near or past the ends of the fp32 range (or a zero vector): the
    // sum again with the vector scaled by the power of two that brings its
    // largest magnitude to [1, 2); this thread's largest magnitude, then its
    // scaled sum of squares
    auto reload_max = [&]() {
      float m = 0.f;
#pragma unroll
      for (int k = 0; k < E; ++k) {
        const int o = a * M + 32 * k + lane;
        m = fmaxf(m, fabsf(F16 ? __half2float(reinterpret_cast<const __half*>(src)[o]) : reinterpret_cast<const float*>(src)[o]));
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, off));
      return m;
    };
    auto reload_ss = [&](float scale) {
      float q = 0.f;
#pragma unroll
      for (int k = 0; k < E; ++k) {
        const int o = a * M + 32 * k + lane;
        const float v = (F16 ? __half2float(reinterpret_cast<const __half*>(src)[o]) : reinterpret_cast<const float*>(src)[o]) * scale;
        q = fmaf(v, v, q);
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) q += __shfl_xor_sync(kFull, q, off);
      return q;
    };
    auto pow2_unit = [](float m) {
      int e;
      frexpf(m, &e);
      return ldexpf(1.f, 1 - e);
    };
    const int64_t r = base + vloc;
    if constexpr (P == 12) {
      // the Paley stage (z_a = Σ_b H12[a][b]·x_b per column i'), one exchange
#pragma unroll
      for (int k = 0; k < E; ++k) zs[a * M + 32 * k + lane] = x[k];
      if (lane == 0) part[a] = ss;
      __syncthreads();
      float s2 = 0.f;
#pragma unroll
      for (int b = 0; b < 12; ++b) s2 += part[b];
      float s = sqrtf(s2);
      if (!(s2 > 1e-30f && s2 < 1e36f)) {  // the same for every thread of the CTA
        const float m = reload_max();
        if (lane == 0) part[16 + a] = m;
        __syncthreads();
        float mm = 0.f;
#pragma unroll
        for (int b = 0; b < 12; ++b) mm = fmaxf(mm, part[16 + b]);
        const float scale = mm > 0.f ? pow2_unit(mm) : 1.f;
        const float q = reload_ss(scale);
        __syncthreads();
        if (lane == 0) part[16 + a] = q;
        __syncthreads();
        float q2 = 0.f;
#pragma unroll
        for (int b = 0; b < 12; ++b) q2 += part[16 + b];
        s = sqrtf(q2) / scale;
      }
      // the Paley stage: thread T < M takes column i' = T of all twelve blocks
      if (tid < M) {
        float xb[12];
#pragma unroll
        for (int b = 0; b < 12; ++b) xb[b] = zs[b * M + tid];
        const float inv = s > 0.f ? 1.f / s : 0.f;
        // Rows 1-11 of H12 are circulant in the quadratic residues mod 11 (+1
        // at b - a in {1, 3, 4, 5, 9}, -1 elsewhere, -1 at b = 0, +1 at b = a):
        // with T = x_1 + ... + x_11 and z_0 = x_0 + T, z_a = 2(p_a + x_a) - z_0,
        // p_a the sum of x_b over the five residue offsets from a.
        float T = xb[1];
#pragma unroll
        for (int b = 2; b < 12; ++b) T += xb[b];
        const float z0 = xb[0] + T;
#pragma unroll
        for (int aa = 0; aa < 12; ++aa) {
          float acc = z0;
          if (aa > 0) {
            const float pa = ((xb[(aa + 0) % 11 + 1] + xb[(aa + 2) % 11 + 1]) + (xb[(aa + 3) % 11 + 1] + xb[(aa + 4) % 11 + 1])) +
                             xb[(aa + 8) % 11 + 1];
            acc = fmaf(2.f, pa + xb[aa], -z0);
          }
          const float v = acc * inv;  // v = z/s
          const int code = wht_code<BM>(v, p.thr, p.sym != 0);
          cbuf[aa * M + tid] = (unsigned char)(s > 0.f ? code : 0);
        }
      }
      __syncthreads();
      if (r < p.N) {
        const int64_t dv = (r / p.group_rows) * p.group_stride + p.offset + (r % p.group_rows);
        const int nw = (D * BM + 31) >> 5;
        for (int w = tid; w < p.W; w += NW * 32) p.codes[dv * p.W + w] = w < nw ? pack_word<BM>(cbuf, w, D) : 0u;
        if (tid == 0) p.norm[dv] = s;
      }
    } else {
      // P = 1: the warp holds the whole vector
      float s = sqrtf(ss);
      if (!(ss > 1e-30f && ss < 1e36f)) {
        const float m = reload_max();
        const float scale = m > 0.f ? pow2_unit(m) : 1.f;
        s = sqrtf(reload_ss(scale)) / scale;
      }
      const float inv = s > 0.f ? 1.f / s : 0.f;
      unsigned char* cw = cbuf + vloc * D;
#pragma unroll
      for (int k = 0; k < E; ++k) {
        const float v = x[k] * inv;
        const int code = wht_code<BM>(v, p.thr, p.sym != 0);
        cw[32 * k + lane] = (unsigned char)(s > 0.f ? code : 0);
      }
      __syncwarp();
      if (r < p.N) {
        const int64_t dv = (r / p.group_rows) * p.group_stride + p.offset + (r % p.group_rows);
        const int nw = (D * BM + 31) >> 5;
        for (int w = lane; w < p.W; w += 32) p.codes[dv * p.W + w] = w < nw ? pack_word<BM>(cw, w, D) : 0u;
        if (lane == 0) p.norm[dv] = s;
      }
    }
  }
}

bool wht_supported(const DevCtx& c) {
  return c.rot == TQ_ROT_HADAMARD && c.mode == TQ_MSE && c.signs != nullptr && c.had_m >= 32 &&
         c.had_m <= 256 && (c.had_p == 1 || c.had_p == 12);
}

// prime: only the one-time setup (shared-memory limit, CTAs per SM) of both
// input types, done when the context is created so that no launch, captured
// into a graph or not, depends on when the first one ran
template <int BM, int P, int E>
static cudaError_t launch_wht_t(const WhtParams& p, bool f16, cudaStream_t st, bool prime = false) {
  constexpr int NW = P == 12 ? 12 : 8, VPC = P == 12 ? 1 : 8, D = P * 32 * E;
  const int64_t ctas = (p.N + VPC - 1) / VPC;
  const size_t smem = (size_t)(P == 12 ? D : 0) * 4 + 32 * 4 + (size_t)((VPC * D + 15) / 16) * 16 +
                      (size_t)kWhtStages * VPC * D * (f16 ? 2 : 4);
  // CTAs resident per SM (registers and shared memory decide), asked once
  // before any stream capture: every CTA of the grid strides over the rows
  // with an equal share, so the grid must fit in one wave
  static PerDeviceValue attr[2], per_sm[2];  // once per device
  if (prime && !f16) {
    const cudaError_t e16 = launch_wht_t<BM, P, E>(p, true, st, true);
    if (e16 != cudaSuccess) return e16;
  }
  const void* kf = f16 ? (const void*)encode_wht_kernel<BM, P, E, true> : (const void*)encode_wht_kernel<BM, P, E, false>;
  const cudaError_t e = smem_attr_once(attr[f16 ? 1 : 0], kf, 160 * 1024);
  if (e != cudaSuccess) return e;
  const int resident = ctas_per_sm_once(per_sm[f16 ? 1 : 0], kf, NW * 32, smem);
  if (prime) return cudaSuccess;
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(ctas, (int64_t)num_sms() * resident));
  if (f16)
    encode_wht_kernel<BM, P, E, true><<<grid, NW * 32, smem, st>>>(p);
  else
    encode_wht_kernel<BM, P, E, false><<<grid, NW * 32, smem, st>>>(p);
  return cudaGetLastError();
}

template <int BM, int P>
static cudaError_t launch_wht_e(const WhtParams& p, bool f16, cudaStream_t st, bool prime) {
  switch (p.m) {
    case 32: return launch_wht_t<BM, P, 1>(p, f16, st, prime);
    case 64: return launch_wht_t<BM, P, 2>(p, f16, st, prime);
    case 128: return launch_wht_t<BM, P, 4>(p, f16, st, prime);
    case 256: return launch_wht_t<BM, P, 8>(p, f16, st, prime);
  }
  return cudaErrorInvalidValue;
}

template <int BM>
static cudaError_t launch_wht_b(const WhtParams& p, int P, bool f16, cudaStream_t st, bool prime = false) {
  return P == 12 ? launch_wht_e<BM, 12>(p, f16, st, prime) : launch_wht_e<BM, 1>(p, f16, st, prime);
}

tq_status prime_encode_wht(const DevCtx& c) {
  if (!wht_supported(c)) return TQ_OK;
  WhtParams p{};
  p.m = c.had_m;
  cudaError_t e = cudaErrorInvalidValue;
  switch (c.b_mse) {
    case 1: e = launch_wht_b<1>(p, c.had_p, false, nullptr, true); break;
    case 2: e = launch_wht_b<2>(p, c.had_p, false, nullptr, true); break;
    case 3: e = launch_wht_b<3>(p, c.had_p, false, nullptr, true); break;
    case 4: e = launch_wht_b<4>(p, c.had_p, false, nullptr, true); break;
    default: return TQ_OK;
  }
  return e == cudaSuccess ? TQ_OK : set_cuda_error(e);
}

tq_status launch_encode_wht(const DevCtx& c, const void* x, int x_dtype, int64_t N, const tq_codes* out,
                            int64_t offset, int64_t group_rows, int64_t group_stride, cudaStream_t stream) {
  if (!wht_supported(c) || out->layout != TQ_LAYOUT_TOKEN) return TQ_ERR_UNSUPPORTED;
  WhtParams p;
  p.x = x;
  p.N = N;
  p.d = c.d;
  p.m = c.had_m;
  p.codes = out->d_codes;
  p.norm = out->d_norm;
  p.W = c.words_per_vec;
  p.signs = c.signs;
  for (int k = 0; k < 15; ++k) p.thr[k] = c.thr[k];
  p.sym = c.sym_thr;
  p.offset = offset;
  p.group_rows = group_rows;
  p.group_stride = group_stride;
  const bool f16 = x_dtype == TQ_F16;
  cudaError_t e = cudaErrorInvalidValue;
  switch (c.b_mse) {
    case 1: e = launch_wht_b<1>(p, c.had_p, f16, stream); break;
    case 2: e = launch_wht_b<2>(p, c.had_p, f16, stream); break;
    case 3: e = launch_wht_b<3>(p, c.had_p, f16, stream); break;
    case 4: e = launch_wht_b<4>(p, c.had_p, f16, stream); break;
    default: return TQ_ERR_UNSUPPORTED;
  }
  return e == cudaSuccess ? TQ_OK : set_cuda_error(e);
}

}  // namespace tq
