// TurboQuant online encoder (MSE and Prod), d <= 128.
//
// One warp encodes 16 vectors; a CTA of 8 warps a tile of 128 vectors.
// Per vector ("TurboQuant 详解", section 一个具体例子 steps 1-6):
//   s = ‖x‖, y = Π·(x/s), idx_i = #{k : √d·y_i >= t_k}, pack, store s.
// The rotation is the dense contraction Y = X·Πᵀ on tensor cores
// (mma.m16n8k16, fp32 accumulation) with operands split into fp16 hi + lo
// parts so that the products carry ~22 significant bits:
//   fp32 input: x·2^e = xh + xl (per-vector power-of-two 2^e, exact), and
//               Y ≈ xh·Πh + xl·Πh + xh·Πl   (3 MMAs)
//   fp16 input: x is exact in fp16, Y ≈ x·Πh + x·Πl  (2 MMAs)
// The output columns are permuted so that lane t of each quad holds the 32
// consecutive coordinates 32t..32t+31 of its two rows: bucketizing and packing
// happen in registers and each lane writes whole words.
//
// TurboQuant_Prod ("TurboQuant 详解", section TurboQuant_prod; "sub-byte-kv-
// cache-quantization-turboquant", section 两阶段量化框架): the same pass runs the
// (b-1)-bit MSE stage, forms r_rot = y - ŷ in registers (γ = ‖r_rot‖ = ‖r‖),
// and a second MMA with the accumulators reused as the A operand computes
// p = (S·Πᵀ)·r_rot = S·r; bit_j = [p_j >= 0].
#include <algorithm>

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {

struct EncParams {
  DevCtx c;
  const void* x;
  int64_t N;
  uint32_t* codes;
  float* norm;
  uint32_t* qjl;
  float* rnorm;
  int layout;
  int W, QW;
  int64_t offset, group_rows, group_stride;
  int pair_aligned;
};

__device__ __forceinline__ int64_t dst_index(const EncParams& p, int64_t r) {
  return (r / p.group_rows) * p.group_stride + p.offset + (r % p.group_rows);
}

// Mask of the bits of pair slot `slot` inside word w of a lane's 2·BM-word
// region of a PAIR block (region starts on a 2·BM-bit boundary).
template <int BM>
__device__ __forceinline__ uint32_t pair_slot_mask(int w, int slot) {
  uint32_t m = 0;
#pragma unroll
  for (int bit = 0; bit < 32; ++bit) {
    int pos = 32 * w + bit;
    if (((pos / BM) & 1) == slot) m |= 1u << bit;
  }
  return m;
}

template <int BM, bool PROD, bool F16>
__global__ void __launch_bounds__(256, 1) encode_kernel(const EncParams p) {
  extern __shared__ __align__(128) uint2 smem[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ int s_abort;
  const int d = p.c.d;
  const int KS = d >> 4;
  constexpr int kFragPerS = 16 * 2 * 32;
  uint2* sPi = smem;
  uint2* sM = smem + 8 * kFragPerS;
  // the operand tables arrive by bulk asynchronous copies (one latency, no
  // per-thread load chains); waits are bounded and report through the status word
  if (threadIdx.x == 0) {
    s_abort = 0;
    mbar_init(&bar, 1);
    fence_mbar_init();
    const uint32_t bpi = (uint32_t)(KS * kFragPerS * sizeof(uint2));
    const uint32_t bm = PROD ? (uint32_t)(8 * kFragPerS * sizeof(uint2)) : 0u;
    mbar_arrive_expect_tx(&bar, bpi + bm);
    bulk_g2s(sPi, p.c.enc_pi, bpi, &bar);
    if (PROD) bulk_g2s(sM, p.c.enc_m, bm, &bar);
  }
  __syncthreads();
  {
    uint32_t spins = 0;
    bool ok = false;
    while (!(ok = mbar_try_wait(&bar, 0)) && ++spins < kSpinLimitDev) {
    }
    if (!ok) {
      atomicOr(p.c.status, 1);
      s_abort = 1;
    }
  }
  __syncthreads();
  if (s_abort) return;  // the copies were waited for (bounded) by every thread above

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const bool lane_valid = 32 * t < d;  // this lane's 32 coordinates exist
  const int64_t ntile = (p.N + 127) / 128;
  constexpr int NCEN = 1 << BM;

  for (int64_t tile = blockIdx.x; tile < ntile; tile += gridDim.x) {
    const int64_t rr[2] = {tile * 128 + warp * 16 + g, tile * 128 + warp * 16 + g + 8};
    // ---------------- load this lane's A elements: cols 16s+2t(+1), 16s+8+2t(+1)
    float xv[8][2][4];
#pragma unroll
    for (int s = 0; s < 8; ++s)
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int q = 0; q < 4; ++q) xv[s][h][q] = 0.f;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if (rr[h] < p.N) {
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          if (s < KS) {
            const int c0 = 16 * s + 2 * t;
            if (F16) {
              const __half2* xr = reinterpret_cast<const __half2*>(
                  static_cast<const __half*>(p.x) + rr[h] * (int64_t)d);
              float2 a = __half22float2(__ldcs(xr + (c0 >> 1)));
              float2 b = __half22float2(__ldcs(xr + ((c0 + 8) >> 1)));
              xv[s][h][0] = a.x; xv[s][h][1] = a.y; xv[s][h][2] = b.x; xv[s][h][3] = b.y;
            } else {
              const float2* xr = reinterpret_cast<const float2*>(
                  static_cast<const float*>(p.x) + rr[h] * (int64_t)d);
              float2 a = __ldcs(xr + (c0 >> 1));
              float2 b = __ldcs(xr + ((c0 + 8) >> 1));
              xv[s][h][0] = a.x; xv[s][h][1] = a.y; xv[s][h][2] = b.x; xv[s][h][3] = b.y;
            }
          }
        }
      }
    }
    // ---------------- a1: norms (lanes 4g..4g+3 share a row)
    float nrm[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float ss = 0.f;
#pragma unroll
      for (int s = 0; s < 8; ++s)
#pragma unroll
        for (int q = 0; q < 4; ++q) ss = fmaf(xv[s][h][q], xv[s][h][q], ss);
      ss += __shfl_xor_sync(kFull, ss, 1);
      ss += __shfl_xor_sync(kFull, ss, 2);
      nrm[h] = sqrtf(ss);
      // squares near or past the ends of the fp32 range (or a zero row): sum
      // them again with the row scaled by the power of two that brings its
      // largest magnitude to [1, 2).  The shuffles run on every lane whenever
      // any lane needs them (the condition differs between rows).
      const bool need = !(ss > 1e-30f && ss < 1e36f);
      if (__any_sync(kFull, need)) {
        float m = 0.f;
#pragma unroll
        for (int s = 0; s < 8; ++s)
#pragma unroll
          for (int q = 0; q < 4; ++q) m = fmaxf(m, fabsf(xv[s][h][q]));
        m = fmaxf(m, __shfl_xor_sync(kFull, m, 1));
        m = fmaxf(m, __shfl_xor_sync(kFull, m, 2));
        float scale = 1.f;
        if (m > 0.f) {
          int e;
          frexpf(m, &e);
          scale = ldexpf(1.f, 1 - e);
        }
        float s2 = 0.f;
#pragma unroll
        for (int s = 0; s < 8; ++s)
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float v = xv[s][h][q] * scale;
            s2 = fmaf(v, v, s2);
          }
        s2 += __shfl_xor_sync(kFull, s2, 1);
        s2 += __shfl_xor_sync(kFull, s2, 2);
        if (need) nrm[h] = sqrtf(s2) / scale;
      }
    }
    // ---------------- a2: rotation on tensor cores
    float sc[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) sc[h] = F16 ? 1.f : pow2_scale_16_32(nrm[h]);
    float acc[16][4];
#pragma unroll
    for (int j = 0; j < 16; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      if (s < KS) {
        uint32_t ah[4], al[4];
        // a0 = (row g, k 2t..), a1 = (row g+8, k 2t..), a2 = (g, k 2t+8..), a3 = (g+8, k 2t+8..)
#pragma unroll
        for (int f = 0; f < 4; ++f) {
          const int h = f & 1, q = (f >> 1) * 2;
          if (F16) {
            ah[f] = pack_f16x2(xv[s][h][q], xv[s][h][q + 1]);  // exact
            al[f] = 0u;
          } else {
            split2(xv[s][h][q] * sc[h], xv[s][h][q + 1] * sc[h], ah[f], al[f]);
          }
        }
        const uint2* bp = sPi + s * kFragPerS;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const uint2 bh = bp[(j * 2 + 0) * 32 + lane];
          const uint2 bl = bp[(j * 2 + 1) * 32 + lane];
          if (!F16) mma16816(acc[j], al[0], al[1], al[2], al[3], bh.x, bh.y);
          mma16816(acc[j], ah[0], ah[1], ah[2], ah[3], bl.x, bl.y);
          mma16816(acc[j], ah[0], ah[1], ah[2], ah[3], bh.x, bh.y);
        }
      }
    }
    // ---------------- a3/a4: bucketize + pack (lane owns coords 32t + l, l = 2j + e)
    uint32_t wd[2][BM];
    float gam[2] = {0.f, 0.f};
    uint32_t qw[2] = {0u, 0u};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
      for (int w = 0; w < BM; ++w) wd[h][w] = 0u;
      const float inv = nrm[h] > 0.f ? p.c.sqrt_d / (nrm[h] * sc[h] * p.c.pi_scale) : 0.f;
#pragma unroll
      for (int j = 0; j < 16; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float v = acc[j][2 * h + e] * inv;
          uint32_t code = 0;
#pragma unroll
          for (int k = 0; k < NCEN - 1; ++k) code += (v >= p.c.thr[k]) ? 1u : 0u;
          if (!(nrm[h] > 0.f) || !lane_valid) code = 0;
          put_bits<BM>(wd[h], (2 * j + e) * BM, code);
          if (PROD) {
            // residual in the rotated domain, unit-vector units: (v - c)/√d
            const float r = (nrm[h] > 0.f && lane_valid) ? (v - p.c.cen[code]) / p.c.sqrt_d : 0.f;
            acc[j][2 * h + e] = r;
            gam[h] = fmaf(r, r, gam[h]);
          }
        }
    }
    // ---------------- a5: QJL stage (Prod)
    if (PROD) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        gam[h] += __shfl_xor_sync(kFull, gam[h], 1);
        gam[h] += __shfl_xor_sync(kFull, gam[h], 2);
        gam[h] = sqrtf(gam[h]);
      }
      const float rs[2] = {pow2_scale_16_32(gam[0]), pow2_scale_16_32(gam[1])};
      float acc2[16][4];
#pragma unroll
      for (int j = 0; j < 16; ++j) acc2[j][0] = acc2[j][1] = acc2[j][2] = acc2[j][3] = 0.f;
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        // K index 16s + 8hh + 2t + e  <->  coordinate 32t + 4s + 2hh + e  (= acc[2s+hh][.. e])
        uint32_t ah[4], al[4];
#pragma unroll
        for (int f = 0; f < 4; ++f) {
          const int row = f & 1, hh = f >> 1;
          const int j = 2 * s + hh;
          split2(acc[j][2 * row] * rs[row], acc[j][2 * row + 1] * rs[row], ah[f], al[f]);
        }
        const uint2* bp = sM + s * kFragPerS;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const uint2 bh = bp[(j * 2 + 0) * 32 + lane];
          const uint2 bl = bp[(j * 2 + 1) * 32 + lane];
          mma16816(acc2[j], al[0], al[1], al[2], al[3], bh.x, bh.y);
          mma16816(acc2[j], ah[0], ah[1], ah[2], ah[3], bl.x, bl.y);
          mma16816(acc2[j], ah[0], ah[1], ah[2], ah[3], bh.x, bh.y);
        }
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t bits = 0;
#pragma unroll
        for (int j = 0; j < 16; ++j)
#pragma unroll
          for (int e = 0; e < 2; ++e) bits |= (acc2[j][2 * h + e] >= 0.f ? 1u : 0u) << (2 * j + e);
        qw[h] = (nrm[h] > 0.f && lane_valid) ? bits : 0u;
        if (!(nrm[h] > 0.f)) gam[h] = 0.f;
      }
    }
    // ---------------- stores
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int64_t r = rr[h];
      const bool have = r < p.N;
      const int64_t dv = have ? dst_index(p, r) : 0;
      if (have && t == 0) {
        p.norm[dv] = nrm[h];
        if (PROD) p.rnorm[dv] = gam[h];
      }
      if (PROD && have && t < p.QW) p.qjl[dv * p.QW + t] = qw[h];
      if (p.layout == TQ_LAYOUT_TOKEN) {
        if (have) {
          uint32_t* dstw = p.codes + dv * p.W + t * BM;
          if (BM == 4) {
            if (t * 4 < p.W) *reinterpret_cast<uint4*>(dstw) = make_uint4(wd[h][0], wd[h][1], wd[h][2], wd[h][3 % BM]);
          } else if (BM == 2) {
            if (t * 2 < p.W) *reinterpret_cast<uint2*>(dstw) = make_uint2(wd[h][0], wd[h][1 % BM]);
          } else {
#pragma unroll
            for (int w = 0; w < BM; ++w)
              if (t * BM + w < p.W) dstw[w] = wd[h][w];
          }
        }
      } else {
        // PAIR layout (d == 128): vector 2i+q's code of coordinate j at bits
        // (2j + q)·BM of block i; this lane owns words [2·BM·t, 2·BM·t + 2·BM).
        const bool even_row = (g & 1) == 0;
        uint32_t part[BM];
#pragma unroll
        for (int w = 0; w < BM; ++w) part[w] = __shfl_down_sync(kFull, wd[h][w], 4);
        const bool partner_here = p.pair_aligned && even_row && (r + 1 < p.N);
        const bool partner_is_writer = p.pair_aligned && !even_row && have;  // written by r-1
        if (have && !partner_is_writer) {
          const int slot = (int)(dv & 1);
          uint32_t* blk = p.codes + (dv >> 1) * (2 * (int64_t)p.W) + 2 * BM * t;
          uint32_t pw[2 * BM];
#pragma unroll
          for (int w = 0; w < 2 * BM; ++w) pw[w] = 0u;
#pragma unroll
          for (int l = 0; l < 32; ++l) {
            const uint32_t cs = get_bits<BM>(wd[h], l * BM);
            put_bits<BM>(pw, (2 * l + slot) * BM, cs);
            if (partner_here) put_bits<BM>(pw, (2 * l + 1) * BM, get_bits<BM>(part, l * BM));
          }
          if (partner_here) {
#pragma unroll
            for (int w = 0; w < 2 * BM; ++w) blk[w] = pw[w];
          } else {
#pragma unroll
            for (int w = 0; w < 2 * BM; ++w) {
              const uint32_t m = pair_slot_mask<BM>(w, slot);
              atomicAnd(blk + w, ~m);
              atomicOr(blk + w, pw[w] & m);
            }
          }
        }
      }
    }
  }
}

template <int BM, bool PROD>
static cudaError_t launch_typed(const EncParams& p, bool f16, int grid, size_t smem,
                                cudaStream_t st) {
  // kernel attributes are set once per device (outside any stream capture that follows)
  static PerDeviceValue attr[2];
  cudaError_t e;
  if (f16) {
    auto k = encode_kernel<BM, PROD, true>;
    e = smem_attr_once(attr[1], (const void*)k, 16 * 16 * 2 * 32 * 8);
    if (e != cudaSuccess) return e;
    k<<<grid, 256, smem, st>>>(p);
  } else {
    auto k = encode_kernel<BM, PROD, false>;
    e = smem_attr_once(attr[0], (const void*)k, 16 * 16 * 2 * 32 * 8);
    if (e != cudaSuccess) return e;
    k<<<grid, 256, smem, st>>>(p);
  }
  return cudaGetLastError();
}

tq_status launch_encode(const DevCtx& c, const void* x, int x_dtype, int64_t N, const tq_codes* out,
                        int64_t offset, int64_t group_rows, int64_t group_stride,
                        cudaStream_t stream) {
  if (out->layout == TQ_LAYOUT_PAIR && c.d != 128) return TQ_ERR_UNSUPPORTED;
  EncParams p;
  p.c = c;
  p.x = x;
  p.N = N;
  p.codes = out->d_codes;
  p.norm = out->d_norm;
  p.qjl = out->d_qjl;
  p.rnorm = out->d_rnorm;
  p.layout = out->layout;
  p.W = c.words_per_vec;
  p.QW = c.qjl_words_per_vec;
  p.offset = offset;
  p.group_rows = group_rows;
  p.group_stride = group_stride;
  p.pair_aligned = (offset % 2 == 0) && (group_rows % 2 == 0 || group_rows >= N) &&
                   (group_stride % 2 == 0);
  const int64_t tiles = (N + 127) / 128;
  const int grid = (int)std::min<int64_t>(tiles, (int64_t)num_sms() * 1);
  const size_t frag = (size_t)16 * 2 * 32 * sizeof(uint2);
  const size_t smem = (c.mode == TQ_PROD ? 16 : (c.d / 16)) * frag;
  const bool f16 = x_dtype == TQ_F16;
  cudaError_t e = cudaErrorInvalidValue;
  const bool prod = c.mode == TQ_PROD;
  switch (c.b_mse) {
    case 1: e = prod ? launch_typed<1, true>(p, f16, grid, smem, stream)
                     : launch_typed<1, false>(p, f16, grid, smem, stream); break;
    case 2: e = prod ? launch_typed<2, true>(p, f16, grid, smem, stream)
                     : launch_typed<2, false>(p, f16, grid, smem, stream); break;
    case 3: e = prod ? launch_typed<3, true>(p, f16, grid, smem, stream)
                     : launch_typed<3, false>(p, f16, grid, smem, stream); break;
    case 4: e = launch_typed<4, false>(p, f16, grid, smem, stream); break;
    default: return TQ_ERR_UNSUPPORTED;
  }
  return e == cudaSuccess ? TQ_OK : set_cuda_error(e);
}

}  // namespace tq
