// Inner-product scores over TurboQuant codes (d = 128).
//
// "sub-byte-kv-cache-quantization-turboquant", section 工程实现的关键路径: the
// query is rotated once (q̂ = Π·q) so that each key costs a table lookup and a
// dot product.  Here the dot products of a 16-key tile with up to 64 queries
// run on tensor cores (mma.m16n8k16): the A operand is built in registers from
// the packed codes through a shared-memory pair table (two coordinates per
// lookup, fp16 values α·c_k), the B operand is q̂/α.
//   MSE : score = s · ⟨q̂, ŷ⟩ = s · Σ_i q̂_i c[idx_i] / √d
//   Prod: + s · γ · √(π/2)/d · Σ_j (S q)_j (2·bit_j − 1)        ("TurboQuant 详解",
//         section TurboQuant_prod; "turboquant-first-principles-walkthrough",
//         section 内积偏差问题与 QJL 修正器), with ±1 A operands built from the
//         sign bits.
// Lane t of each quad reads the 32 consecutive coordinates 32t..32t+31 of its
// two keys (whole words); the MMA K index is permuted to match:
//   K index 16s + 8h + 2t + e  <->  coordinate 32t + 4s + 2h + e.
#include <algorithm>

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {

constexpr int kQTile = 64;  // queries per launch of the scan kernel

// Query preparation, one block (8 warps) per query: q̂ = Π·q / α and, for
// Prod, S·q, computed with coalesced float4 row loads (warp w: rows
// 16w..16w+15), then written as B fragments (uint2 per lane):
//   b0 = (K index 16s+2t.., col g), b1 = (16s+8+2t.., col g),
//   K index 16s+8h+2t+e <-> coordinate 32t+4s+2h+e, query = 8·tile + g.
// ws layout: [mse | qjl] x [qtile][kstep][lane] uint2.
__device__ __forceinline__ float warp_dot4(float4 a, float4 b) {
  float x = a.x * b.x + a.y * b.y + a.z * b.z + a.w * b.w;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(kFull, x, o);
  return x;
}

__global__ void __launch_bounds__(256) scores_qprep_kernel(const DevCtx c, const float* __restrict__ q, int M,
                                                           uint2* __restrict__ frag_mse,
                                                           uint2* __restrict__ frag_qjl) {
  const int m = blockIdx.x;
  __shared__ float qs[128], qr[128], sq[128];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid < 128) qs[tid] = (m < M) ? q[(int64_t)m * 128 + tid] : 0.f;
  __syncthreads();
  const float4 qq = *reinterpret_cast<const float4*>(&qs[4 * lane]);
  const bool prod = c.mode == TQ_PROD;
  float4 pv[16];
#pragma unroll
  for (int r = 0; r < 16; ++r)
    pv[r] = __ldg(reinterpret_cast<const float4*>(c.pi + (size_t)(16 * warp + r) * 128) + lane);
#pragma unroll
  for (int r = 0; r < 16; ++r) {
    const float x = warp_dot4(pv[r], qq);
    if (lane == 0) qr[16 * warp + r] = x / c.alpha;
  }
  if (prod) {
#pragma unroll
    for (int r = 0; r < 16; ++r)
      pv[r] = __ldg(reinterpret_cast<const float4*>(c.s_mat + (size_t)(16 * warp + r) * 128) + lane);
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      const float x = warp_dot4(pv[r], qq);
      if (lane == 0) sq[16 * warp + r] = x;
    }
  }
  __syncthreads();
  if (tid < 32) {
    const int s = tid >> 2, t = tid & 3, g = m & 7, nt = m >> 3;
    const int ln = 4 * g + t;
    const int c0 = 32 * t + 4 * s, c1 = c0 + 2;
    uint2 f;
    f.x = pack_f16x2(qr[c0], qr[c0 + 1]);
    f.y = pack_f16x2(qr[c1], qr[c1 + 1]);
    frag_mse[((size_t)nt * 8 + s) * 32 + ln] = f;
    if (prod) {
      f.x = pack_f16x2(sq[c0], sq[c0 + 1]);
      f.y = pack_f16x2(sq[c1], sq[c1 + 1]);
      frag_qjl[((size_t)nt * 8 + s) * 32 + ln] = f;
    }
  }
}

struct ScoreParams {
  DevCtx c;
  const uint32_t* codes;
  const float* norm;
  const uint32_t* qjl;
  const float* rnorm;
  int64_t first, N;
  int W, QW;
  const uint2* frag_mse;  // this launch's query tiles
  const uint2* frag_qjl;
  int m0, mq;             // first query, queries in this launch (<= 64)
  int M;                  // total queries (row count of scores)
  float* scores;
};

template <int BM, bool PROD>
__global__ void __launch_bounds__(256, 2) scores_kernel(const ScoreParams p) {
  extern __shared__ uint32_t sh[];
  constexpr int E = 1 << (2 * BM);
  uint32_t* lut = sh;                             // [E][32] replicated per lane
  uint2* fm = reinterpret_cast<uint2*>(sh + E * 32);  // [8 qtiles][8 ksteps][32]
  uint2* fq = fm + 8 * 8 * 32;
  const int nqt = (p.mq + 7) >> 3;
  for (int i = threadIdx.x; i < E * 32; i += blockDim.x) lut[i] = p.c.lut[i >> 5];
  for (int i = threadIdx.x; i < nqt * 8 * 32; i += blockDim.x) {
    fm[i] = p.frag_mse[i];
    if (PROD) fq[i] = p.frag_qjl[i];
  }
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const uint32_t* mylut = lut + lane;
  const float inv_sd = 1.f / p.c.sqrt_d;
  const float qjl_c = 1.2533141373155001f / (float)p.c.d;  // √(π/2)/d
  const int64_t ntile = (p.N + 15) >> 4;
  for (int64_t tile = (int64_t)blockIdx.x * 8 + warp; tile < ntile; tile += (int64_t)gridDim.x * 8) {
    const int64_t k0 = tile * 16 + g, k1 = k0 + 8;
    const bool h0 = k0 < p.N, h1 = k1 < p.N;
    uint32_t w0[BM], w1[BM];
#pragma unroll
    for (int w = 0; w < BM; ++w) {
      w0[w] = h0 ? __ldcs(p.codes + (p.first + k0) * p.W + t * BM + w) : 0u;
      w1[w] = h1 ? __ldcs(p.codes + (p.first + k1) * p.W + t * BM + w) : 0u;
    }
    uint32_t qb0 = 0, qb1 = 0;
    float g0 = 0.f, g1 = 0.f;
    if (PROD) {
      qb0 = h0 ? __ldcs(p.qjl + (p.first + k0) * p.QW + t) : 0u;
      qb1 = h1 ? __ldcs(p.qjl + (p.first + k1) * p.QW + t) : 0u;
      g0 = h0 ? p.rnorm[p.first + k0] : 0.f;
      g1 = h1 ? p.rnorm[p.first + k1] : 0.f;
    }
    const float s0 = h0 ? p.norm[p.first + k0] : 0.f;
    const float s1 = h1 ? p.norm[p.first + k1] : 0.f;
    float acc[8][4], acq[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[n][e] = acq[n][e] = 0.f;
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      const uint32_t a0 = mylut[get_bits<2 * BM>(w0, 4 * s * BM) << 5];
      const uint32_t a1 = mylut[get_bits<2 * BM>(w1, 4 * s * BM) << 5];
      const uint32_t a2 = mylut[get_bits<2 * BM>(w0, (4 * s + 2) * BM) << 5];
      const uint32_t a3 = mylut[get_bits<2 * BM>(w1, (4 * s + 2) * BM) << 5];
      uint32_t c0 = 0, c1 = 0, c2 = 0, c3 = 0;
      if (PROD) {
        // ±1 from sign bits: bit 1 -> +1 (0x3C00), bit 0 -> -1 (0xBC00)
        const uint32_t y0 = ~(qb0 >> (4 * s)), y1 = ~(qb1 >> (4 * s));
        c0 = 0x3C003C00u | ((y0 & 1u) << 15) | ((y0 & 2u) << 30);
        c1 = 0x3C003C00u | ((y1 & 1u) << 15) | ((y1 & 2u) << 30);
        c2 = 0x3C003C00u | ((y0 & 4u) << 13) | ((y0 & 8u) << 28);
        c3 = 0x3C003C00u | ((y1 & 4u) << 13) | ((y1 & 8u) << 28);
      }
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        if (n < nqt) {
          const uint2 b = fm[(n * 8 + s) * 32 + lane];
          mma16816(acc[n], a0, a1, a2, a3, b.x, b.y);
          if (PROD) {
            const uint2 bq = fq[(n * 8 + s) * 32 + lane];
            mma16816(acq[n], c0, c1, c2, c3, bq.x, bq.y);
          }
        }
      }
    }
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      if (n < nqt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int qi = 8 * n + 2 * t + (e & 1);
          const bool hi = e >= 2;
          const int64_t key = hi ? k1 : k0;
          if (qi < p.mq && key < p.N) {
            const float s = hi ? s1 : s0;
            float v = acc[n][e] * inv_sd;
            if (PROD) v = fmaf((hi ? g1 : g0) * qjl_c, acq[n][e], v);
            p.scores[(int64_t)(p.m0 + qi) * p.N + key] = s * v;
          }
        }
      }
    }
  }
}

size_t scores_ws_bytes(const DevCtx& c, int M) {
  size_t tiles = (size_t)(M + 7) / 8;
  return tiles * 8 * 32 * sizeof(uint2) * 2 + 256;
}

template <int BM, bool PROD>
static cudaError_t run_scores(ScoreParams p, cudaStream_t st) {
  constexpr int E = 1 << (2 * BM);
  const size_t smem = (size_t)E * 32 * 4 + 2 * 8 * 8 * 32 * sizeof(uint2);
  auto k = scores_kernel<BM, PROD>;
  static int attr_done = 0;  // set once, outside any later stream capture
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_done = 1;
  }
  const int64_t tiles = (p.N + 15) / 16;
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>((tiles + 7) / 8, (int64_t)num_sms() * 4));
  k<<<grid, 256, smem, st>>>(p);
  return cudaGetLastError();
}

tq_status launch_scores(const DevCtx& c, const float* q, int M, const tq_codes* keys, int64_t first,
                        int64_t N, float* scores, void* ws, size_t ws_bytes, cudaStream_t stream) {
  const size_t tiles = (size_t)(M + 7) / 8;
  uint2* fm = static_cast<uint2*>(ws);
  uint2* fq = fm + tiles * 8 * 32;
  scores_qprep_kernel<<<(int)(tiles * 8), 256, 0, stream>>>(c, q, M, fm, fq);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_cuda_error(e);
  ScoreParams p;
  p.c = c;
  p.codes = keys->d_codes;
  p.norm = keys->d_norm;
  p.qjl = keys->d_qjl;
  p.rnorm = keys->d_rnorm;
  p.first = first;
  p.N = N;
  p.W = c.words_per_vec;
  p.QW = c.qjl_words_per_vec;
  p.M = M;
  p.scores = scores;
  const bool prod = c.mode == TQ_PROD;
  for (int m0 = 0; m0 < M; m0 += kQTile) {
    p.m0 = m0;
    p.mq = std::min(kQTile, M - m0);
    p.frag_mse = fm + (size_t)(m0 / 8) * 8 * 32;
    p.frag_qjl = fq + (size_t)(m0 / 8) * 8 * 32;
    switch (c.b_mse) {
      case 1: e = prod ? run_scores<1, true>(p, stream) : run_scores<1, false>(p, stream); break;
      case 2: e = prod ? run_scores<2, true>(p, stream) : run_scores<2, false>(p, stream); break;
      case 3: e = prod ? run_scores<3, true>(p, stream) : run_scores<3, false>(p, stream); break;
      case 4: e = run_scores<4, false>(p, stream); break;
      default: return TQ_ERR_UNSUPPORTED;
    }
    if (e != cudaSuccess) return set_cuda_error(e);
  }
  return TQ_OK;
}

}  // namespace tq
