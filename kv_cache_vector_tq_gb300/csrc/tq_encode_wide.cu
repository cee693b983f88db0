// TurboQuant_MSE encoder for wide vectors (d = 128·C, C >= 2) with a dense
// rotation: the contraction Y = X·Πᵀ as a tiled GEMM on tensor cores.
//
// "TurboQuant 详解", section 一个具体例子 steps 1-6 (per vector: s = ‖x‖,
// y = Π·x/s, idx_i = #{k : √d·y_i >= t_k}, pack, store s); the rotation is
// the one dense matrix product of the encoder ("turboquant-first-principles-
// walkthrough", section 通用码本设计: encoding is one matmul and one lookup).
//
// A CTA owns 128 rows x 64 output coordinates (8 warps x 16 rows; the 64
// coordinates are half of a 128-coordinate chunk of the encoder's operand
// table, so lane t of a quad ends with 16 consecutive coordinates of its two
// rows).  The K loop runs over 128-wide chunks of x, double-buffered in shared
// memory by cp.async together with the matching slice of the fp16 hi/lo
// table of pi_scale·Π.  Per chunk and row, x is scaled by a power of two
// chosen from the chunk's own norm before the hi/lo split (no range
// assumption on the input), the three products xh·Πh + xl·Πh + xh·Πl
// accumulate in fp32 over the chunk only, and the chunk result joins a
// float-float running sum: over K = 3072 a single fp32 accumulator would
// carry errors of several 1e-7 in unit-variance units, too close to the 1e-6
// band around the codebook thresholds.  The epilogue bucketizes and packs in
// registers.
#include <algorithm>

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {

namespace {

struct WideParams {
  const void* x;
  int64_t N;
  int d, W;
  uint32_t* codes;
  float* norm;
  const uint2* frag;  // pi_scale·Π, fp16 hi/lo: ((c·KS + s)·16 + j)·2 + plane)·32 + lane
  float pi_scale, sqrt_d;
  float thr[15];
  int64_t offset, group_rows, group_stride;
};

constexpr int kRowStride = 136;  // elements per staged row (128 + 8: conflict-free fragment reads)
constexpr int kBBytes = 8 * 8 * 2 * 32 * 8;  // 8 k-steps x 8 n-tiles x hi/lo x 32 lanes x uint2

__device__ __forceinline__ void cp16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_wait1() { asm volatile("cp.async.wait_group 1;\n" ::: "memory"); }

__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = a + b;
  const float bb = s - a;
  e = (a - (s - bb)) + (b - bb);
}

template <int BM, bool F16>
__global__ void __launch_bounds__(256, 1) encode_wide_kernel(const WideParams p) {
  constexpr int ES = F16 ? 2 : 4;                   // bytes per input element
  constexpr int ABytes = 128 * kRowStride * ES;      // one staged chunk of x
  constexpr int Stage = ABytes + kBBytes;
  constexpr int PPR = 128 * ES / 16;                 // 16-byte pieces per row chunk
  constexpr int WPL = BM / 2;                        // code words per lane per row (16 codes)
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g = lane >> 2, t = lane & 3;
  const int nkc = p.d / 128, KS = p.d / 16, ncb = p.d / 64;
  const int64_t ntiles = (p.N + 127) / 128;

  for (int64_t item = blockIdx.x; item < ntiles * ncb; item += gridDim.x) {
    const int64_t rt = item / ncb;
    const int cb = (int)(item % ncb), c = cb >> 1, hf = cb & 1;
    const int64_t row0 = rt * 128;

    auto load_chunk = [&](int kc, int st) {
      unsigned char* A = smem + st * Stage;
      unsigned char* Bs = A + ABytes;
      for (int i = tid; i < 128 * PPR; i += 256) {
        const int r = i / PPR, q = i % PPR;
        unsigned char* dst = A + r * kRowStride * ES + q * 16;
        if (row0 + r < p.N)
          cp16(dst, static_cast<const unsigned char*>(p.x) + ((row0 + r) * p.d + kc * 128) * ES + q * 16);
        else
          *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
      }
      // table slice: k-steps kc·8 .. +7, n-tiles 8hf .. 8hf+7 (4 KB contiguous per k-step)
      for (int i = tid; i < kBBytes / 16; i += 256) {
        const int s = i >> 8, q = i & 255;
        const uint2* src = p.frag + (((int64_t)c * KS + kc * 8 + s) * 16 + 8 * hf) * 2 * 32;
        cp16(Bs + s * 4096 + q * 16, reinterpret_cast<const unsigned char*>(src) + q * 16);
      }
      cp_commit();
    };
    auto ld2 = [&](const unsigned char* A, int r, int col) -> float2 {
      if constexpr (F16)
        return __half22float2(*reinterpret_cast<const __half2*>(A + (r * kRowStride + col) * 2));
      else
        return *reinterpret_cast<const float2*>(A + (r * kRowStride + col) * 4);
    };

    float run_hi[8][4], run_lo[8][4];
#pragma unroll
    for (int jj = 0; jj < 8; ++jj)
#pragma unroll
      for (int e = 0; e < 4; ++e) run_hi[jj][e] = run_lo[jj][e] = 0.f;
    double ss_a = 0.0, ss_b = 0.0;  // rows g and g+8 of this warp
    const int ra = 16 * warp + g, rb = ra + 8;

    load_chunk(0, 0);
    for (int kc = 0; kc < nkc; ++kc) {
      if (kc + 1 < nkc)
        load_chunk(kc + 1, (kc + 1) & 1);
      else
        cp_commit();
      cp_wait1();
      __syncthreads();
      const unsigned char* A = smem + (kc & 1) * Stage;
      const uint2* Bs = reinterpret_cast<const uint2*>(A + ABytes);
      // the chunk's norm per row (this lane's 32 elements, then the quad)
      float sa = 0.f, sb = 0.f;
#pragma unroll
      for (int s = 0; s < 8; ++s)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const float2 u = ld2(A, ra, 16 * s + 8 * hh + 2 * t), w = ld2(A, rb, 16 * s + 8 * hh + 2 * t);
          sa = fmaf(u.y, u.y, fmaf(u.x, u.x, sa));
          sb = fmaf(w.y, w.y, fmaf(w.x, w.x, sb));
        }
      sa += __shfl_xor_sync(kFull, sa, 1);
      sa += __shfl_xor_sync(kFull, sa, 2);
      sb += __shfl_xor_sync(kFull, sb, 1);
      sb += __shfl_xor_sync(kFull, sb, 2);
      ss_a += (double)sa;
      ss_b += (double)sb;
      const float sca = pow2_scale_16_32(sqrtf(sa)), scb = pow2_scale_16_32(sqrtf(sb));
      float acc[8][4];
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) acc[jj][0] = acc[jj][1] = acc[jj][2] = acc[jj][3] = 0.f;
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const float2 x0 = ld2(A, ra, 16 * s + 2 * t), x1 = ld2(A, rb, 16 * s + 2 * t);
        const float2 x2 = ld2(A, ra, 16 * s + 8 + 2 * t), x3 = ld2(A, rb, 16 * s + 8 + 2 * t);
        uint32_t ah[4], al[4];
        split2(x0.x * sca, x0.y * sca, ah[0], al[0]);
        split2(x1.x * scb, x1.y * scb, ah[1], al[1]);
        split2(x2.x * sca, x2.y * sca, ah[2], al[2]);
        split2(x3.x * scb, x3.y * scb, ah[3], al[3]);
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          const uint2 bh = Bs[s * 512 + (jj * 2 + 0) * 32 + lane];
          const uint2 bl = Bs[s * 512 + (jj * 2 + 1) * 32 + lane];
          mma16816(acc[jj], al[0], al[1], al[2], al[3], bh.x, bh.y);
          mma16816(acc[jj], ah[0], ah[1], ah[2], ah[3], bl.x, bl.y);
          mma16816(acc[jj], ah[0], ah[1], ah[2], ah[3], bh.x, bh.y);
        }
      }
      // undo the chunk's power-of-two scale (exact) and add into the float-float sums
      const float ia = 1.f / sca, ib = 1.f / scb;
#pragma unroll
      for (int jj = 0; jj < 8; ++jj)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float sum, err;
          two_sum(run_hi[jj][e], acc[jj][e] * (e < 2 ? ia : ib), sum, err);
          run_hi[jj][e] = sum;
          run_lo[jj][e] += err;
        }
      __syncthreads();  // everyone is done with this stage before it is refilled
    }

    // ---- epilogue: s, bucketize, pack (lane t: coordinates 128c + 32t + 16hf + 0..15)
    const float s_a = (float)sqrt(ss_a), s_b = (float)sqrt(ss_b);
    const float inv_a = s_a > 0.f ? p.sqrt_d / (s_a * p.pi_scale) : 0.f;
    const float inv_b = s_b > 0.f ? p.sqrt_d / (s_b * p.pi_scale) : 0.f;
    uint32_t wa[WPL], wb[WPL];
#pragma unroll
    for (int w = 0; w < WPL; ++w) wa[w] = wb[w] = 0u;
#pragma unroll
    for (int jj = 0; jj < 8; ++jj)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float va = (run_hi[jj][e] + run_lo[jj][e]) * inv_a;
        const float vb = (run_hi[jj][2 + e] + run_lo[jj][2 + e]) * inv_b;
        uint32_t ca = 0, cbk = 0;
#pragma unroll
        for (int k = 0; k < (1 << BM) - 1; ++k) {
          ca += va >= p.thr[k] ? 1u : 0u;
          cbk += vb >= p.thr[k] ? 1u : 0u;
        }
        if (!(s_a > 0.f)) ca = 0;
        if (!(s_b > 0.f)) cbk = 0;
        const int pos = (2 * jj + e) * BM;
        wa[pos >> 5] |= ca << (pos & 31);
        wb[pos >> 5] |= cbk << (pos & 31);
      }
    const int word0 = ((128 * c + 32 * t + 16 * hf) * BM) >> 5;
    const int64_t rows[2] = {row0 + ra, row0 + rb};
    const float ns[2] = {s_a, s_b};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int64_t r = rows[h];
      if (r < p.N) {
        const int64_t dv = (r / p.group_rows) * p.group_stride + p.offset + (r % p.group_rows);
#pragma unroll
        for (int w = 0; w < WPL; ++w) p.codes[dv * p.W + word0 + w] = h ? wb[w] : wa[w];
        if (cb == 0 && t == 0) p.norm[dv] = ns[h];
      }
    }
  }
}

template <int BM>
cudaError_t launch_wide_t(const WideParams& p, bool f16, cudaStream_t st) {
  const int64_t items = (p.N + 127) / 128 * (p.d / 64);
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(items, (int64_t)num_sms()));
  static int attr_done[2] = {0, 0};  // set once, before any stream capture
  if (f16) {
    constexpr size_t smem = 2 * (128 * kRowStride * 2 + kBBytes);
    auto k = encode_wide_kernel<BM, true>;
    if (!attr_done[1]) {
      cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      attr_done[1] = 1;
    }
    k<<<grid, 256, smem, st>>>(p);
  } else {
    constexpr size_t smem = 2 * (128 * kRowStride * 4 + kBBytes);
    auto k = encode_wide_kernel<BM, false>;
    if (!attr_done[0]) {
      cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      attr_done[0] = 1;
    }
    k<<<grid, 256, smem, st>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace

bool wide_supported(const DevCtx& c) {
  return c.d > kChunk && c.d % kChunk == 0 && c.mode == TQ_MSE && (c.b_mse == 2 || c.b_mse == 4);
}

tq_status launch_encode_wide(const DevCtx& c, const void* x, int x_dtype, int64_t N, const tq_codes* out,
                             int64_t offset, int64_t group_rows, int64_t group_stride, cudaStream_t stream) {
  if (!wide_supported(c) || out->layout != TQ_LAYOUT_TOKEN) return TQ_ERR_UNSUPPORTED;
  WideParams p;
  p.x = x;
  p.N = N;
  p.d = c.d;
  p.W = c.words_per_vec;
  p.codes = out->d_codes;
  p.norm = out->d_norm;
  p.frag = c.enc_pi;
  p.pi_scale = c.pi_scale;
  p.sqrt_d = c.sqrt_d;
  for (int k = 0; k < 15; ++k) p.thr[k] = c.thr[k];
  p.offset = offset;
  p.group_rows = group_rows;
  p.group_stride = group_stride;
  const bool f16 = x_dtype == TQ_F16;
  const cudaError_t e = c.b_mse == 4 ? launch_wide_t<4>(p, f16, stream) : launch_wide_t<2>(p, f16, stream);
  return e == cudaSuccess ? TQ_OK : set_cuda_error(e);
}

}  // namespace tq
