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
// Work split: m threads per vector (m in 32..256), 256/m vectors per CTA;
// thread i' holds element a·m + i' of each of the P blocks a.  The Sylvester
// stages pair threads i' and i' ^ h: by warp shuffles for h < 32, through
// shared memory above; the 12 x 12 Paley stage is a fixed signed sum of the
// thread's own P values.  Plain fp32 butterflies: each output sees one
// rounding per stage, so the error in v stays near √(log2 d)·2^-24 (about
// 2e-7 at d = 3072), inside the 1e-6 band around the codebook thresholds.
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

template <int BM, int P, bool F16>
__global__ void __launch_bounds__(256) encode_wht_kernel(const WhtParams p) {
  extern __shared__ __align__(16) float wsm[];  // [256/m vectors][P][m], then the norm partials
  const int m = p.m;
  const int vpc = 256 / m;  // vectors per CTA
  const int tid = threadIdx.x, lane = tid & 31;
  const int vloc = tid / m, ip = tid % m;  // vector within the CTA, element index within a block
  float* my = wsm + vloc * P * m;
  float* red = wsm + vpc * P * m;  // [8 warps]
  float sg[P];
#pragma unroll
  for (int a = 0; a < P; ++a) sg[a] = p.signs[a * m + ip];

  for (int64_t base = (int64_t)blockIdx.x * vpc; base < p.N; base += (int64_t)gridDim.x * vpc) {
    const int64_t r = base + vloc;
    const bool have = r < p.N;
    float x[P];
#pragma unroll
    for (int a = 0; a < P; ++a) {
      float v = 0.f;
      if (have) {
        const int64_t o = r * p.d + a * m + ip;
        v = F16 ? __half2float(__ldcs(static_cast<const __half*>(p.x) + o)) : __ldcs(static_cast<const float*>(p.x) + o);
      }
      x[a] = v;
    }
    // s = ‖x‖: the thread's P squares, then a tree over the vector's m threads
    float ss = 0.f;
#pragma unroll
    for (int a = 0; a < P; ++a) ss = fmaf(x[a], x[a], ss);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(kFull, ss, off);
    if (m > 32) {
      __syncthreads();  // the previous vector's readers of red are done
      if (lane == 0) red[tid >> 5] = ss;
      __syncthreads();
      ss = 0.f;
      for (int w = 0; w < m / 32; ++w) ss += red[vloc * (m / 32) + w];
    }
    const float s = sqrtf(ss);
    // σ ∘ x, then the Sylvester stages over i'
#pragma unroll
    for (int a = 0; a < P; ++a) x[a] *= sg[a];
    for (int h = 1; h < m; h <<= 1) {
      if (h < 32) {
#pragma unroll
        for (int a = 0; a < P; ++a) {
          const float o = __shfl_xor_sync(kFull, x[a], h);
          x[a] = (ip & h) ? (o - x[a]) : (x[a] + o);
        }
      } else {
        __syncthreads();
#pragma unroll
        for (int a = 0; a < P; ++a) my[a * m + ip] = x[a];
        __syncthreads();
#pragma unroll
        for (int a = 0; a < P; ++a) {
          const float o = my[a * m + (ip ^ h)];
          x[a] = (ip & h) ? (o - x[a]) : (x[a] + o);
        }
      }
    }
    // the Paley stage across the blocks: z_a = Σ_b H12[a][b]·x_b
    float z[P];
    if constexpr (P == 12) {
#pragma unroll
      for (int a = 0; a < 12; ++a) {
        float acc = 0.f;
#pragma unroll
        for (int bb = 0; bb < 12; ++bb) acc = paley12_sign(a, bb) > 0 ? acc + x[bb] : acc - x[bb];
        z[a] = acc;
      }
    } else {
#pragma unroll
      for (int a = 0; a < P; ++a) z[a] = x[a];
    }
    // bucketize v = z/s and pack: the 32 coordinates of a warp's lanes share BM words
    const float inv = s > 0.f ? 1.f / s : 0.f;
    const int64_t dv = have ? (r / p.group_rows) * p.group_stride + p.offset + (r % p.group_rows) : 0;
#pragma unroll
    for (int a = 0; a < P; ++a) {
      const float v = z[a] * inv;
      uint32_t code = 0;
#pragma unroll
      for (int k = 0; k < (1 << BM) - 1; ++k) code += v >= p.thr[k] ? 1u : 0u;
      if (!(s > 0.f)) code = 0;
      const int pos = lane * BM;  // bit position within the 32-coordinate group
      uint32_t w[BM];
#pragma unroll
      for (int k = 0; k < BM; ++k) {
        uint32_t c = 0;
        if ((pos >> 5) == k) c = code << (pos & 31);
        if ((pos >> 5) + 1 == k && (pos & 31) + BM > 32) c = code >> (32 - (pos & 31));
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) c |= __shfl_xor_sync(kFull, c, off);
        w[k] = c;
      }
      if (have && lane < BM) {
        // group of coordinates a·m + 32q .. +31, q = i' / 32: words from (a·m + 32q)·BM / 32
        const int word0 = ((a * m + (ip & ~31)) * BM) >> 5;
        uint32_t val = w[0];
#pragma unroll
        for (int k = 1; k < BM; ++k)
          if (lane == k) val = w[k];
        p.codes[dv * p.W + word0 + lane] = val;
      }
    }
    if (have && ip == 0) {
      p.norm[dv] = s;
      for (int w = (p.d * BM + 31) / 32; w < p.W; ++w) p.codes[dv * p.W + w] = 0u;
    }
  }
}

bool wht_supported(const DevCtx& c) {
  return c.rot == TQ_ROT_HADAMARD && c.mode == TQ_MSE && c.signs != nullptr && c.had_m >= 32 &&
         c.had_m <= 256 && (c.had_p == 1 || c.had_p == 12);
}

template <int BM, int P>
static cudaError_t launch_wht_t(const WhtParams& p, bool f16, cudaStream_t st) {
  const int vpc = 256 / p.m;
  const int64_t ctas = (p.N + vpc - 1) / vpc;
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(ctas, (int64_t)num_sms() * 8));
  const size_t smem = ((size_t)vpc * P * p.m + 8) * sizeof(float);
  if (f16)
    encode_wht_kernel<BM, P, true><<<grid, 256, smem, st>>>(p);
  else
    encode_wht_kernel<BM, P, false><<<grid, 256, smem, st>>>(p);
  return cudaGetLastError();
}

template <int BM>
static cudaError_t launch_wht_b(const WhtParams& p, int P, bool f16, cudaStream_t st) {
  return P == 12 ? launch_wht_t<BM, 12>(p, f16, st) : launch_wht_t<BM, 1>(p, f16, st);
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
