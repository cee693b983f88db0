// TurboQuant_MSE encoder for wide vectors (d = 128·C, C >= 2) with a dense
// rotation, on the fifth-generation tensor cores (tcgen05.mma, accumulators in
// tensor memory).
//
// "TurboQuant 详解", section 一个具体例子 steps 1-6 (per vector: s = ‖x‖,
// y = Π·x/s, idx_i = #{k : √d·y_i >= t_k}, pack, store s); the rotation is
// the one dense matrix product of the encoder ("turboquant-first-principles-
// walkthrough", section 通用码本设计: encoding is one matmul and one lookup).
//
// Two launches.
//  1. row_norm_kernel: s = ‖x‖ per row (fp32 sums of 8 squares, fp64 across
//     them), stored as the code set's norm.
//  2. encode_umma_kernel: a persistent CTA per SM walks tiles of 128 rows x
//     128 output coordinates; K runs in 64-wide chunks.
//
// Precision.  A code must agree with the fp64 definition outside a 1e-6 band
// around each threshold.  Rows are scaled by a power of two (s·sc in [16, 32))
// and split into fp16 hi + lo; pi_scale·Π is split the same way on the host;
// the products xl·Πh + xh·Πl (one accumulator over all of K) and xh·Πh (two
// accumulators, one per half of K) carry about 22 bits of each operand.  The
// tensor cores' fp32 accumulation truncates: measured on GB300 its error in v
// units grows linearly with the length L of the accumulated K range (largest
// error over 1.3e5 outputs about 7e-9·L, biased toward zero: ~1e-5 for a
// 1536-long range) — far above the band.  So the epilogue flags every
// coordinate whose v lies within m = max(5e-6, 6e-8·L) of a threshold (about
// nine times the largest measured error) and recomputes it: one warp forms
// Σ_k x_k·Π_jk in float-float arithmetic from the input row and the fp32 copy
// of Π (error ~3e-8 in v units) and decides the code again.  The flagged
// fraction is about 2m·Σ_k pdf(t_k): ~7e-4 of the coordinates at d = 3072,
// b = 4, one or two per row.
//
// Warp roles (14 warps):
//   0-7   converters: thread = row = TMEM lane, K half = warp / 4.  Reads its
//         row's 32 elements of the staged chunk, writes the fp16 hi and lo
//         pairs into a tensor-memory A stage (the MMA's A operand).
//   8-11  epilogue: thread = row.  First sums the three accumulators into v
//         and writes v over H1, which frees the low-order accumulator and H0
//         for the next tile at once; then bucketizes from H1 (freeing it before
//         the next tile reaches its second half of K), refines, packs, stores.
//   12    producer: one 2-D TMA load per chunk of the x tile (128 rows, boxes
//         of 128 bytes per row in the 128-byte swizzle, so that 32 threads
//         reading one 16-byte column of 32 rows hit every bank once per 8
//         rows) and one 32 KB bulk copy of the Π tile (hi and lo planes in
//         core-matrix order).
//   13    MMA issuer (one thread): per chunk 12 tcgen05.mma of M = 128,
//         N = 128, K = 16, A from tensor memory, B from shared memory.
// Tensor memory (512 columns x 128 lanes): A stages at columns 0-127
// (2 x [hi 32 | lo 32]), the low-order accumulator at 128, H0 at 256, H1 at 384.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {

namespace {

constexpr int kTM = 128;                     // rows per tile (TMEM lanes)
constexpr int kTN = kUmmaTN;                 // output coordinates per tile (MMA N)
constexpr int kKC = kUmmaKC;                 // K per chunk
constexpr int kStages = 3;                   // x / Π stages in shared memory
constexpr int kAStages = 2;                  // A stages in tensor memory
constexpr int kBPlane = kUmmaPlaneBytes;     // one fp16 plane of a Π tile: 16 KB
constexpr int kBStage = 2 * kBPlane;         // hi + lo
constexpr int kThreads = 14 * 32;
constexpr uint32_t kColLo = 128, kColH0 = 256, kColH1 = 384;
constexpr int kCodeRow = kTN + 4;
constexpr int kRefineBatch = 6;  // bytes per row of the epilogue's code buffer (rows on distinct banks)

template <bool F16>
struct XLayout {
  static constexpr int ES = F16 ? 2 : 4;
  static constexpr int BoxCols = 128 / ES;       // one TMA box: 128 rows x 128 bytes
  static constexpr int Boxes = kKC / BoxCols;    // per chunk: 2 (fp32) or 1 (fp16)
  static constexpr int Stage = kTM * kKC * ES;   // 1024-byte aligned (swizzle atom)
  static constexpr int Smem = kStages * kBStage + kStages * Stage + kTM * kCodeRow + 256;
};

struct UmmaParams {
  const void* x;
  int64_t N;
  int d, W;
  uint32_t* codes;
  const float* norm;          // filled by row_norm_kernel
  const unsigned char* btab;  // pi_scale·Π tiles: ((ob·nkc + kc)·2 + plane)·16 KB, core-matrix order
  const float* pi;            // Π, fp32 row-major (refinement)
  float pi_scale, margin;
  double sqrt_d;
  float thr[15];
  int64_t offset, group_rows, group_stride;
  int* status;
  uint32_t wait_limit;
};

__device__ __forceinline__ int64_t dest_row(int64_t r, int64_t offset, int64_t group_rows, int64_t group_stride) {
  return (r / group_rows) * group_stride + offset + (r % group_rows);
}

// ------------------------------------------------------------------ pass 1: row norms
template <bool F16>
__global__ void __launch_bounds__(256) row_norm_kernel(const void* x, int64_t N, int d, float* norm, int64_t offset,
                                                       int64_t group_rows, int64_t group_stride) {
  const int lane = threadIdx.x & 31;
  const int64_t w0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t r = w0; r < N; r += nw) {
    double ss = 0.0;
    if constexpr (F16) {
      const uint4* row = reinterpret_cast<const uint4*>(static_cast<const __half*>(x) + r * d);
      for (int k = lane; k < d / 8; k += 32) {
        const uint4 u = __ldg(row + k);
        const __half2* h = reinterpret_cast<const __half2*>(&u);
        float acc = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 f = __half22float2(h[j]);
          acc = fmaf(f.x, f.x, acc);
          acc = fmaf(f.y, f.y, acc);
        }
        ss += (double)acc;
      }
    } else {
      const float4* row = reinterpret_cast<const float4*>(static_cast<const float*>(x) + r * d);
      const int n4 = d / 4;
      for (int k = lane; k < n4; k += 64) {
        const float4 a = __ldg(row + k);
        float acc = fmaf(a.x, a.x, fmaf(a.y, a.y, fmaf(a.z, a.z, a.w * a.w)));
        if (k + 32 < n4) {
          const float4 b = __ldg(row + k + 32);
          acc = fmaf(b.x, b.x, fmaf(b.y, b.y, fmaf(b.z, b.z, fmaf(b.w, b.w, acc))));
        }
        ss += (double)acc;
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(kFull, ss, o);
    if (!(ss > 1e-30 && ss < 1e36)) {
      // squares near or past the ends of the fp32 range (or a zero row): sum
      // them again with the row scaled by the power of two that brings its
      // largest magnitude to [1, 2)
      float m = 0.f;
      for (int k = lane; k < d; k += 32)
        m = fmaxf(m, fabsf(F16 ? __half2float(static_cast<const __half*>(x)[r * d + k]) : static_cast<const float*>(x)[r * d + k]));
#pragma unroll
      for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
      if (m > 0.f) {
        int e;
        frexpf(m, &e);
        const float sc = ldexpf(1.f, 1 - e);
        double s2 = 0.0;
        for (int k = lane; k < d; k += 32) {
          const float v = (F16 ? __half2float(static_cast<const __half*>(x)[r * d + k]) : static_cast<const float*>(x)[r * d + k]) * sc;
          s2 += (double)(v * v);
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) s2 += __shfl_xor_sync(kFull, s2, o);
        ss = s2 / ((double)sc * (double)sc);
      } else {
        ss = 0.0;
      }
    }
    if (lane == 0) norm[dest_row(r, offset, group_rows, group_stride)] = (float)sqrt(ss);
  }
}

// ------------------------------------------------------------------ pass 2: GEMM, bucketize, pack
template <int BM, bool F16>
__global__ void __launch_bounds__(kThreads, 1) encode_umma_kernel(const UmmaParams p,
                                                                   const __grid_constant__ CUtensorMap xmap) {
  using XL = XLayout<F16>;
  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char* sB = smem;
  unsigned char* sX = smem + kStages * kBStage;
  unsigned char* sCodes = sX + kStages * XL::Stage;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sCodes + kTM * kCodeRow);
  uint64_t* x_full = bars;
  uint64_t* x_empty = bars + 3;
  uint64_t* b_full = bars + 6;
  uint64_t* b_empty = bars + 9;
  uint64_t* a_full = bars + 12;
  uint64_t* a_empty = bars + 14;
  uint64_t* acc_full = bars + 16;
  uint64_t* acc_empty_a = bars + 17;  // low-order accumulator and H0 free
  uint64_t* acc_empty_b = bars + 18;  // H1 free
  uint64_t* drain = bars + 19;
  float* thr_s = reinterpret_cast<float*>(bars + 20);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(thr_s + 16);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nkc = p.d / kKC, nob = p.d / kTN;
  const int64_t ntiles = (p.N + kTM - 1) / kTM * nob;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&x_full[s], 1);
      mbar_init(&x_empty[s], 8);
      mbar_init(&b_full[s], 1);
      mbar_init(&b_empty[s], 1);
    }
    for (int s = 0; s < kAStages; ++s) {
      mbar_init(&a_full[s], 8);
      mbar_init(&a_empty[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty_a, 4);
    mbar_init(acc_empty_b, 4);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (tid < 16) thr_s[tid] = tid < (1 << BM) - 1 ? p.thr[tid] : INFINITY;
  if (warp == 0) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 8) {
    // ---------------- converters
    const int q = warp & 3, hh = warp >> 2, rl = 32 * q + lane;
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;
    uint32_t i = 0;
    bool ok = true;
    for (int64_t t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
      const int64_t row = t / nob * kTM + rl;
      const bool valid = row < p.N;
      const float s = valid ? p.norm[dest_row(row, p.offset, p.group_rows, p.group_stride)] : 0.f;
      const float sc = pow2_scale_16_32(s);
      for (int kc = 0; kc < nkc; ++kc, ++i) {
        const uint32_t xs = i % kStages;
        if (!__all_sync(kFull, bar_wait(&x_full[xs], (i / kStages) & 1u, abort_flag, p.status, p.wait_limit))) {
          ok = false;
          break;
        }
        float v[32];
        if (valid) {
          // 16-byte column c of row rl sits at column c ^ (rl % 8) of the 128-byte row
          const int sw = rl & 7;
          if constexpr (F16) {
            const unsigned char* src = sX + xs * XL::Stage + rl * 128;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint4 u = *reinterpret_cast<const uint4*>(src + 16 * ((4 * hh + j) ^ sw));
              const __half2* h = reinterpret_cast<const __half2*>(&u);
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float2 f = __half22float2(h[e]);
                v[8 * j + 2 * e] = f.x;
                v[8 * j + 2 * e + 1] = f.y;
              }
            }
          } else {
            const unsigned char* src = sX + xs * XL::Stage + hh * (kTM * 128) + rl * 128;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float4 f = *reinterpret_cast<const float4*>(src + 16 * (j ^ sw));
              v[4 * j] = f.x;
              v[4 * j + 1] = f.y;
              v[4 * j + 2] = f.z;
              v[4 * j + 3] = f.w;
            }
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = 0.f;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&x_empty[xs]);
        uint32_t hi[16], lo[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) split2(v[2 * j] * sc, v[2 * j + 1] * sc, hi[j], lo[j]);
        const uint32_t as = i % kAStages;
        if (!__all_sync(kFull, bar_wait(&a_empty[as], ((i / kAStages) & 1u) ^ 1u, abort_flag, p.status, p.wait_limit))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t col = as * 64 + 16 * hh;
        tmem_st16(tmem + lane_base + col, hi);
        tmem_st16(tmem + lane_base + col + 32, lo);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&a_full[as]);
      }
    }
  } else if (warp < 12) {
    // ---------------- epilogue
    const int q = warp & 3, rl = 32 * q + lane;
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;
    uint32_t tl = 0;
    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, ++tl) {
      const int64_t rt = t / nob;
      const int ob = (int)(t % nob);
      const int64_t row = rt * kTM + rl;
      const bool valid = row < p.N;
      if (!__all_sync(kFull, bar_wait(acc_full, tl & 1u, abort_flag, p.status, p.wait_limit))) break;
      tc_fence_after();
      const int64_t dv = valid ? dest_row(row, p.offset, p.group_rows, p.group_stride) : 0;
      const float s = valid ? p.norm[dv] : 0.f;
      const float sc = pow2_scale_16_32(s);
      const float f = s > 0.f ? (float)(p.sqrt_d / ((double)s * sc * p.pi_scale)) : 0.f;
      // phase 1: v = (H0 + H1 + Lo)·f written over H1; Lo and H0 go back to the MMA
#pragma unroll 1
      for (int g = 0; g < 8; ++g) {
        uint32_t a[16], b[16], c[16];
        tmem_ld16_nw(tmem + lane_base + kColLo + 16 * g, a);
        tmem_ld16_nw(tmem + lane_base + kColH0 + 16 * g, b);
        tmem_ld16_nw(tmem + lane_base + kColH1 + 16 * g, c);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j)
          c[j] = __float_as_uint(((__uint_as_float(b[j]) + __uint_as_float(c[j])) + __uint_as_float(a[j])) * f);
        tmem_st16(tmem + lane_base + kColH1 + 16 * g, c);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty_a);
      // phase 2: bucketize from H1; codes of this row one byte per coordinate
      // (refined in place, packed at the end)
      unsigned char* my_codes = sCodes + rl * kCodeRow;
      uint32_t fm[4] = {0u, 0u, 0u, 0u};
#pragma unroll 1
      for (int g = 0; g < 8; ++g) {  // 16 columns at a time
        uint32_t c[16];
        tmem_ld16_nw(tmem + lane_base + kColH1 + 16 * g, c);
        tmem_wait_ld();
        uint32_t m16 = 0u, packed[4];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          bool near;
          const uint32_t code = bucketize<BM>(__uint_as_float(c[j]), thr_s, p.margin, near);
          if ((j & 3) == 0) packed[j >> 2] = 0u;
          packed[j >> 2] |= code << (8 * (j & 3));
          m16 |= (near ? 1u : 0u) << j;
        }
#pragma unroll
        for (int w = 0; w < 4; ++w) reinterpret_cast<uint32_t*>(my_codes + 16 * g)[w] = packed[w];
        const uint32_t part = m16 << (16 * (g & 1));
        if (g < 2)
          fm[0] |= part;
        else if (g < 4)
          fm[1] |= part;
        else if (g < 6)
          fm[2] |= part;
        else
          fm[3] |= part;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty_b);
      if (!(valid && s > 0.f)) fm[0] = fm[1] = fm[2] = fm[3] = 0u;

      // refinement of the flagged coordinates, one warp-wide dot product each
      for (;;) {
        const uint32_t any = __ballot_sync(kFull, (fm[0] | fm[1] | fm[2] | fm[3]) != 0u);
        if (!any) break;
        const int src = __ffs(any) - 1;
        int col = 0;
        if (lane == src) {
#pragma unroll
          for (int g = 3; g >= 0; --g)
            if (fm[g]) col = 32 * g + __ffs(fm[g]) - 1;
#pragma unroll
          for (int g = 0; g < 4; ++g)
            if (g == (col >> 5)) fm[g] &= fm[g] - 1u;
        }
        col = __shfl_sync(kFull, col, src);
        const int64_t srow = rt * kTM + 32 * q + src;
        const float* prow = p.pi + (int64_t)(ob * kTN + col) * p.d;
        float sh = 0.f, sl = 0.f;
        // kRefineBatch loads of each operand in flight per lane
        for (int k0 = 4 * lane; k0 < p.d; k0 += 128 * kRefineBatch) {
          float4 xv[kRefineBatch], pv[kRefineBatch];
#pragma unroll
          for (int u = 0; u < kRefineBatch; ++u) {
            const int k = k0 + 128 * u;
            if (k < p.d) {
              pv[u] = __ldg(reinterpret_cast<const float4*>(prow + k));
              if constexpr (F16) {
                const uint2 h = __ldg(reinterpret_cast<const uint2*>(static_cast<const __half*>(p.x) + srow * p.d + k));
                const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&h.x));
                const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&h.y));
                xv[u] = make_float4(a.x, a.y, b.x, b.y);
              } else {
                xv[u] = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(p.x) + srow * p.d + k));
              }
            }
          }
#pragma unroll
          for (int u = 0; u < kRefineBatch; ++u) {
            if (k0 + 128 * u < p.d) {
              ff_fma(xv[u].x, pv[u].x, sh, sl);
              ff_fma(xv[u].y, pv[u].y, sh, sl);
              ff_fma(xv[u].z, pv[u].z, sh, sl);
              ff_fma(xv[u].w, pv[u].w, sh, sl);
            }
          }
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
          const float oh = __shfl_xor_sync(kFull, sh, o), ol = __shfl_xor_sync(kFull, sl, o);
          const float s2 = sh + oh, bb = s2 - sh;
          sl = sl + ol + ((sh - (s2 - bb)) + (oh - bb));
          sh = s2;
        }
        if (lane == src) {
          const float vv = (float)(((double)sh + (double)sl) * (p.sqrt_d / (double)s));
          bool near;
          my_codes[col] = (unsigned char)bucketize<BM>(vv, thr_s, 0.f, near);
        }
      }

      if (valid) {
        uint32_t wd[4 * BM];
#pragma unroll
        for (int w = 0; w < 4 * BM; ++w) wd[w] = 0u;
        if (s > 0.f) {
#pragma unroll
          for (int w = 0; w < kTN / 4; ++w) {
            const uint32_t four = reinterpret_cast<const uint32_t*>(my_codes)[w];
#pragma unroll
            for (int e = 0; e < 4; ++e) put_bits<BM>(wd, (4 * w + e) * BM, (four >> (8 * e)) & 0xFFu);
          }
        }
        uint4* dst = reinterpret_cast<uint4*>(p.codes + dv * p.W + (int64_t)ob * (4 * BM));
#pragma unroll
        for (int w = 0; w < BM; ++w) dst[w] = make_uint4(wd[4 * w], wd[4 * w + 1], wd[4 * w + 2], wd[4 * w + 3]);
      }
    }
  } else if (warp == 12) {
    // ---------------- producer
    uint32_t i = 0;
    bool ok = true;
    const uint64_t pol_b = l2_policy_evict_last();
    for (int64_t t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
      const int64_t row0 = t / nob * kTM;
      const int ob = (int)(t % nob);
      for (int kc = 0; kc < nkc; ++kc, ++i) {
        const uint32_t s = i % kStages, ph = ((i / kStages) & 1u) ^ 1u;
        if (!__all_sync(kFull, bar_wait(&x_empty[s], ph, abort_flag, p.status, p.wait_limit) &&
                                   bar_wait(&b_empty[s], ph, abort_flag, p.status, p.wait_limit))) {
          ok = false;
          break;
        }
        if (lane == 0) {
          // rows past N read as zeros and still count toward the box's bytes
          mbar_arrive_expect_tx(&x_full[s], (uint32_t)XL::Stage);
          mbar_arrive_expect_tx(&b_full[s], (uint32_t)kBStage);
          // the Π tiles are read by every CTA again and again: keep them in L2
          // (a row tile is read once per output block by CTAs that run about
          // together, so the rows take the default policy: marked evict-first
          // they were fetched from DRAM again for every block)
#pragma unroll
          for (int bx = 0; bx < XL::Boxes; ++bx)
            tma_load_2d(sX + s * XL::Stage + bx * (kTM * 128), &xmap, kc * kKC + bx * XL::BoxCols, (int)row0,
                        &x_full[s]);
          bulk_g2s_hint(sB + s * kBStage, p.btab + ((int64_t)ob * nkc + kc) * kBStage, kBStage, &b_full[s], pol_b);
        }
        __syncwarp();
      }
    }
    if (!ok && lane == 0) {
      // copies still in flight land before the CTA may exit (bounded)
      for (uint32_t j = i >= (uint32_t)kStages ? i - kStages : 0u; j < i; ++j) {
        for (uint32_t n = 0; n < kSpinLimitDev && !mbar_try_wait(&x_full[j % kStages], (j / kStages) & 1u); ++n) {
        }
        for (uint32_t n = 0; n < kSpinLimitDev && !mbar_try_wait(&b_full[j % kStages], (j / kStages) & 1u); ++n) {
        }
      }
    }
  } else if (lane == 0) {
    // ---------------- MMA issuer
    const uint32_t idesc = umma_idesc_f16(kTM, kTN);
    uint32_t i = 0, tl = 0;
    bool ok = true;
    for (int64_t t = blockIdx.x; t < ntiles && ok; t += gridDim.x, ++tl) {
      if (!bar_wait(acc_empty_a, (tl & 1u) ^ 1u, abort_flag, p.status, p.wait_limit)) break;
      tc_fence_after();
      for (int kc = 0; kc < nkc; ++kc, ++i) {
        const uint32_t s = i % kStages, as = i % kAStages;
        if (kc == nkc / 2 && !bar_wait(acc_empty_b, (tl & 1u) ^ 1u, abort_flag, p.status, p.wait_limit)) {
          ok = false;
          break;
        }
        if (!bar_wait(&b_full[s], (i / kStages) & 1u, abort_flag, p.status, p.wait_limit) ||
            !bar_wait(&a_full[as], (i / kAStages) & 1u, abort_flag, p.status, p.wait_limit)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t bbase = smem_u32(sB + s * kBStage);
        const uint32_t hcol = kc < nkc / 2 ? kColH0 : kColH1;
        const bool first_h = kc == 0 || kc == nkc / 2;
#pragma unroll
        for (int ks = 0; ks < kKC / 16; ++ks) {
          const uint64_t bh = umma_desc(bbase + ks * 256, 128, 1024);
          const uint64_t bl = umma_desc(bbase + kBPlane + ks * 256, 128, 1024);
          const uint32_t ah = tmem + as * 64 + 8 * ks, al = ah + 32;
          umma_f16_ts(tmem + kColLo, al, bh, idesc, (kc | ks) != 0 ? 1u : 0u);
          umma_f16_ts(tmem + kColLo, ah, bl, idesc, 1u);
          umma_f16_ts(tmem + hcol, ah, bh, idesc, (first_h && ks == 0) ? 0u : 1u);
        }
        umma_commit(&b_empty[s]);
        umma_commit(&a_empty[as]);
      }
      if (ok) umma_commit(acc_full);
    }
    // every MMA issued has completed before tensor memory is released (bounded)
    umma_commit(drain);
    for (uint32_t n = 0; n < kSpinLimitDev && !mbar_try_wait(drain, 0u); ++n) {
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int BM, bool F16>
cudaError_t launch_umma_t(const UmmaParams& p, const CUtensorMap& xmap, cudaStream_t st) {
  auto k = encode_umma_kernel<BM, F16>;
  static PerDeviceValue attr;  // set once per device, before any stream capture
  const cudaError_t e = smem_attr_once(attr, (const void*)k, XLayout<F16>::Smem);
  if (e != cudaSuccess) return e;
  const int64_t tiles = (p.N + kTM - 1) / kTM * (p.d / kTN);
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(tiles, (int64_t)num_sms()));
  k<<<grid, kThreads, XLayout<F16>::Smem, st>>>(p, xmap);
  return cudaGetLastError();
}

template <bool F16>
cudaError_t launch_bm(const UmmaParams& p, const CUtensorMap& xmap, int bm, cudaStream_t st) {
  switch (bm) {
    case 1: return launch_umma_t<1, F16>(p, xmap, st);
    case 2: return launch_umma_t<2, F16>(p, xmap, st);
    case 3: return launch_umma_t<3, F16>(p, xmap, st);
    default: return launch_umma_t<4, F16>(p, xmap, st);
  }
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (the library
// does not link the driver library itself).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

}  // namespace

tq_status rows_tensor_map(CUtensorMap* map, const void* x, int64_t N, int d, bool f16) {
  const int es = f16 ? 2 : 4;
  const cuuint64_t gdim[2] = {(cuuint64_t)d, (cuuint64_t)N};
  const cuuint64_t gstride[1] = {(cuuint64_t)d * es};
  const cuuint32_t box[2] = {(cuuint32_t)(128 / es), (cuuint32_t)kTM};
  const cuuint32_t estride[2] = {1u, 1u};
  const PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (!encode) return TQ_ERR_CUDA;
  const CUresult r = encode(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
                            const_cast<void*>(x), gdim, gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? TQ_OK : TQ_ERR_INVALID_ARG;
}

bool umma_supported(const DevCtx& c) {
  return c.d > kChunk && c.d % kTN == 0 && c.mode == TQ_MSE && c.b_mse >= 1 && c.b_mse <= 4 && c.umma_tab != nullptr;
}

tq_status launch_encode_umma(const DevCtx& c, const void* x, int x_dtype, int64_t N, const tq_codes* out,
                             int64_t offset, int64_t group_rows, int64_t group_stride, cudaStream_t stream) {
  if (!umma_supported(c) || out->layout != TQ_LAYOUT_TOKEN) return TQ_ERR_UNSUPPORTED;
  if (N > INT32_MAX) return TQ_ERR_UNSUPPORTED;  // TMA row coordinates are 32-bit
  const bool f16 = x_dtype == TQ_F16;
  {
    // one warp per row, 8 rows per CTA in flight; as many CTAs as are resident
    // at once (each warp strides over the rows with an equal share)
    static PerDeviceValue per_sm[2];  // asked once per device, before any stream capture
    const int resident = f16 ? ctas_per_sm_once(per_sm[1], (const void*)row_norm_kernel<true>, 256, 0)
                             : ctas_per_sm_once(per_sm[0], (const void*)row_norm_kernel<false>, 256, 0);
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>((N + 7) / 8, (int64_t)num_sms() * resident));
    if (f16)
      row_norm_kernel<true><<<grid, 256, 0, stream>>>(x, N, c.d, out->d_norm, offset, group_rows, group_stride);
    else
      row_norm_kernel<false><<<grid, 256, 0, stream>>>(x, N, c.d, out->d_norm, offset, group_rows, group_stride);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return set_cuda_error(e);
  }
  UmmaParams p;
  p.x = x;
  p.N = N;
  p.d = c.d;
  p.W = c.words_per_vec;
  p.codes = out->d_codes;
  p.norm = out->d_norm;
  p.btab = c.umma_tab;
  p.pi = c.pi;
  p.pi_scale = c.pi_scale;
  p.sqrt_d = std::sqrt((double)c.d);
  p.margin = std::max(5e-6f, 6e-8f * (float)(c.d / 2));
  for (int k = 0; k < 15; ++k) p.thr[k] = c.thr[k];
  p.offset = offset;
  p.group_rows = group_rows;
  p.group_stride = group_stride;
  p.status = c.status;
  p.wait_limit = c.wait_limit;
  CUtensorMap xmap;
  const tq_status ms = rows_tensor_map(&xmap, x, N, c.d, f16);
  if (ms != TQ_OK) return ms;
  const cudaError_t e =
      f16 ? launch_bm<true>(p, xmap, c.b_mse, stream) : launch_bm<false>(p, xmap, c.b_mse, stream);
  return e == cudaSuccess ? TQ_OK : set_cuda_error(e);
}

}  // namespace tq
