// Split-sequence decode attention over a TurboQuant_MSE KV cache (d = 128).
//
// "TurboQuant 详解", section decode 阶段到底怎么“用”这些压缩后的 KV (second
// route): the kernel unpacks, looks up, scales and consumes the codes inside
// attention, never materialising fp16 K/V.  "sub-byte-kv-cache-quantization-
// turboquant", section 工程实现的关键路径: the query is rotated once and every
// query head reads kv_head = q_head / (Hq / Hkv).
//
// Per (batch, kv head) the token range is cut into work items; a persistent
// CTA takes an item, pulls its K codes, V pair blocks and norms into shared
// memory with bulk asynchronous copies completing on one mbarrier, and its 8
// warps process 16-token tiles:
//   K side  S[t][n] = Σ_κ K̂[t][κ]·Q[κ][n]      (mma.m16n8k16, A built from a
//           shared-memory pair table, B = pre-rotated queries, hi/lo columns)
//   softmax online per head, base-2 logits with the scale folded into Q
//   V side  O[μ][n] += Σ_t V̂[μ][t]·W[t][n]     (A from V pair blocks, which
//           hold the codes of two consecutive tokens side by side; B = p·s_v)
// O stays in the rotated domain: Σ_t p_t s_t Πᵀŷ_t = Πᵀ Σ_t p_t s_t ŷ_t, so the
// merge kernel applies Πᵀ once per head after combining the splits with the
// usual log-sum-exp rule.
#include <algorithm>
#include <mutex>
#include <utility>

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {

constexpr int kTileTok = 16;
constexpr int kDecWarps = 8;
// resident split CTAs per SM (register budget: 2 for up to 4 heads per KV head, 1 for 8)
static int ctas_per_sm(int G) { return G >= 8 ? 1 : 2; }
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLazy = 8.f;          // rescale only when the max grows by > 2^8

struct DecPlan {
  int S;           // splits (work items) per (batch, kv head)
  int tiles;       // tiles per (batch, kv head)
  int per_item;    // tiles per item (last one may have fewer)
  int NT;          // 8-column n-tiles (2·G columns)
};

static DecPlan make_plan(int B, int Hq, int Hkv, int64_t seq) {
  DecPlan pl;
  pl.tiles = (int)((seq + kTileTok - 1) / kTileTok);
  const int groups = std::max(1, B * Hkv);
  const int G = Hkv > 0 ? Hq / Hkv : 1;
  const int ctas = ctas_per_sm(G) * num_sms();
  int S = std::max(1, (ctas + groups - 1) / groups);
  S = std::min(S, pl.tiles);
  pl.per_item = (pl.tiles + S - 1) / S;
  pl.S = (pl.tiles + pl.per_item - 1) / pl.per_item;
  pl.NT = (2 * G + 7) / 8;
  return pl;
}

size_t decode_ws_bytes(int d, int B, int Hq, int Hkv, int64_t seq) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || seq <= 0) return 256;
  DecPlan pl = make_plan(B, Hq, Hkv, seq);
  size_t frag = (size_t)B * Hkv * 8 * pl.NT * 32 * sizeof(uint2);
  size_t part = (size_t)B * Hq * pl.S * (2 + 128) * sizeof(float);
  return (frag + 255) / 256 * 256 + part + 256;
}

// ------------------------------------------------------------------ query prep
// One block (8 warps) per (batch, kv head): q̂_h = Π·q_h for the G query heads
// of the group, folded with scale·log2(e)/(√d·α_K) and split into fp16 hi
// (column 2h) and lo (column 2h+1) B fragments: b0 = (K index 16s+2t.., col g),
// b1 = (16s+8+2t.., col g), K index 16s+8h+2t+e <-> coordinate 32t+4s+2h+e.
// Warp w computes rows 16w..16w+15 of Π·q with coalesced float4 loads of Π.
__global__ void __launch_bounds__(256) decode_qprep_kernel(const float* __restrict__ pi,
                                                           const void* __restrict__ q, int q_f16,
                                                           int Hq, int G, int NT, float fold,
                                                           uint2* __restrict__ frag) {
  __shared__ float qs[8][128];
  __shared__ float qr[8][128];
  const int bk = blockIdx.x;  // b * Hkv + kvh
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int Hkv = Hq / G;
  const int b = bk / Hkv, kvh = bk % Hkv;
  float4 pv[16];
#pragma unroll
  for (int r = 0; r < 16; ++r)
    pv[r] = __ldg(reinterpret_cast<const float4*>(pi + (size_t)(16 * warp + r) * 128) + lane);
  griddep_wait();  // q and the workspace may be produced / still read by earlier grids
  for (int e = tid; e < G * 128; e += blockDim.x) {
    const int h = e >> 7, i = e & 127;
    const int64_t off = ((int64_t)b * Hq + kvh * G + h) * 128 + i;
    qs[h][i] = q_f16 ? __half2float(static_cast<const __half*>(q)[off]) : static_cast<const float*>(q)[off];
  }
  __syncthreads();
  for (int h = 0; h < G; ++h) {
    const float4 qq = *reinterpret_cast<const float4*>(&qs[h][4 * lane]);
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      float x = pv[r].x * qq.x + pv[r].y * qq.y + pv[r].z * qq.z + pv[r].w * qq.w;
      x += __shfl_xor_sync(kFull, x, 16);
      x += __shfl_xor_sync(kFull, x, 8);
      x += __shfl_xor_sync(kFull, x, 4);
      x += __shfl_xor_sync(kFull, x, 2);
      x += __shfl_xor_sync(kFull, x, 1);
      if (lane == 0) qr[h][16 * warp + r] = x * fold;
    }
  }
  __syncthreads();
  griddep_launch();
  // entries: s (8) x nt (NT) x lane (32)
  for (int e = tid; e < 8 * NT * 32; e += blockDim.x) {
    const int ln = e & 31, nt = (e >> 5) % NT, s = e / (32 * NT);
    const int g = ln >> 2, t = ln & 3;
    const int n = nt * 8 + g, h = n >> 1, lo = n & 1;
    uint2 f = make_uint2(0u, 0u);
    if (h < G) {
      const int c0 = 32 * t + 4 * s;
      float v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float x = qr[h][c0 + u];
        const float hi = __half2float(__float2half_rn(x));
        v[u] = lo ? (x - hi) : hi;
      }
      f.x = pack_f16x2(v[0], v[1]);
      f.y = pack_f16x2(v[2], v[3]);
    }
    frag[((size_t)bk * 8 + s) * NT * 32 + nt * 32 + ln] = f;
  }
}

// Word loads as one vector access where the width allows it (4 words are
// 16-byte aligned, 2 words 8-byte aligned, in every layout read here).
// Codes are read once: streaming loads that do not keep the lines in L1.
template <int N>
__device__ __forceinline__ void ldg_words(uint32_t (&w)[N], const uint32_t* src) {
  if constexpr (N == 4) {
    const uint4 v = __ldcs(reinterpret_cast<const uint4*>(src));
    w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
  } else if constexpr (N == 2) {
    const uint2 v = __ldcs(reinterpret_cast<const uint2*>(src));
    w[0] = v.x; w[1] = v.y;
  } else {
#pragma unroll
    for (int i = 0; i < N; ++i) w[i] = __ldcs(src + i);
  }
}

// Shared memory of the split kernel: the pair tables of K (and of V when its
// codebook differs), replicated once per lane so that lookups never conflict,
// and the scratch in which the 8 warps of a CTA combine their softmax states.
struct DecSmem {
  int off_vlut, off_comb, bytes;
};

static DecSmem dec_smem(int bk, int bv, int G, bool same_lut) {
  DecSmem m;
  const int lutk = (1 << (2 * bk)) * 32 * 4, lutv = same_lut ? 0 : (1 << (2 * bv)) * 32 * 4;
  m.off_vlut = lutk;
  m.off_comb = lutk + lutv;
  m.bytes = m.off_comb + kDecWarps * G * 130 * 4;
  return m;
}

// ------------------------------------------------------------------ split kernel
struct DecParams {
  const uint32_t* klut;  // global tables (copied to shared memory)
  const uint32_t* vlut;
  float v_fold;          // 1 / (α_V √d)
  const uint32_t* kcodes;
  const float* knorm;
  const uint32_t* vcodes;
  const float* vnorm;
  int64_t seq, cap;
  int B, Hq, Hkv, G;
  DecPlan pl;
  const uint2* qfrag;
  float* part;           // [B*Hq][S][130]: m, l, acc[128]
  DecSmem sm;
  int same_lut;
};

// One tile's operands, loaded one tile ahead of its use.
template <int BK, int BV>
struct TileRegs {
  uint32_t k0[BK], k1[BK], v0[BV], v1[BV];
  float nk0, nk1, nv0, nv1;
};

template <int BK, int BV>
__device__ __forceinline__ void load_tile(TileRegs<BK, BV>& r, const uint32_t* kb, const uint32_t* vb,
                                          const float* knb, const float* vnb, int lt0, int g, int t) {
  constexpr int WK = 4 * BK, WV = 4 * BV;
  ldg_words<BK>(r.k0, kb + (size_t)(lt0 + g) * WK + t * BK);
  ldg_words<BK>(r.k1, kb + (size_t)(lt0 + g + 8) * WK + t * BK);
  // V pair blocks t and t+4 of the tile (tokens 2t,2t+1 and 2t+8,2t+9); coordinates 16g..16g+15
  ldg_words<BV>(r.v0, vb + (size_t)((lt0 >> 1) + t) * (2 * WV) + g * BV);
  ldg_words<BV>(r.v1, vb + (size_t)((lt0 >> 1) + 4 + t) * (2 * WV) + g * BV);
  r.nk0 = __ldcs(knb + lt0 + g);
  r.nk1 = __ldcs(knb + lt0 + g + 8);
  r.nv0 = __ldcs(vnb + lt0 + g);
  r.nv1 = __ldcs(vnb + lt0 + g + 8);
}

template <int BK, int BV, int G>
__global__ void __launch_bounds__(256, (G >= 8 ? 1 : 2)) decode_split_kernel(const DecParams p) {
  constexpr int NT = (2 * G + 7) / 8;
  constexpr int WK = 4 * BK, WV = 4 * BV;  // words per vector (d = 128)
  constexpr int EK = 1 << (2 * BK), EV = 1 << (2 * BV);
  extern __shared__ __align__(128) unsigned char smem[];
  uint32_t* klut = reinterpret_cast<uint32_t*>(smem);
  uint32_t* vlut = p.same_lut ? klut : reinterpret_cast<uint32_t*>(smem + p.sm.off_vlut);
  float* comb = reinterpret_cast<float*>(smem + p.sm.off_comb);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
#pragma unroll 8
  for (int i = tid; i < EK * 32; i += blockDim.x) klut[i] = __ldg(p.klut + (i >> 5));
  if (!p.same_lut) {
#pragma unroll 8
    for (int i = tid; i < EV * 32; i += blockDim.x) vlut[i] = __ldg(p.vlut + (i >> 5));
  }
  __syncthreads();
  griddep_wait();    // codes (appends), query fragments and partials of earlier grids
  griddep_launch();  // the merge grid may start staging its tables
  const uint32_t* mykl = klut + lane;
  const uint32_t* myvl = vlut + lane;

  const int n_items = p.B * p.Hkv * p.pl.S;
  for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int bk = item / p.pl.S, sp = item % p.pl.S;
    const int tile0 = sp * p.pl.per_item;
    const int ntl = min(p.pl.per_item, p.pl.tiles - tile0);
    const int64_t tok0 = (int64_t)tile0 * kTileTok;
    const int64_t vbase = (int64_t)bk * p.cap + tok0;  // vector index of the item's first token
    const uint32_t* kb = p.kcodes + vbase * WK;
    const uint32_t* vb = p.vcodes + vbase * WV;  // vbase even: pair blocks align
    const float* knb = p.knorm + vbase;
    const float* vnb = p.vnorm + vbase;

    uint2 qf[8][NT];
#pragma unroll
    for (int s = 0; s < 8; ++s)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) qf[s][nt] = p.qfrag[((size_t)bk * 8 + s) * NT * 32 + nt * 32 + lane];
    float m_run[NT], l_run[NT];
    float o[8][NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      m_run[nt] = -INFINITY;
      l_run[nt] = 0.f;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) o[mt][nt][0] = o[mt][nt][1] = o[mt][nt][2] = o[mt][nt][3] = 0.f;
    }

    TileRegs<BK, BV> cur, nxt;
    if (warp < ntl) load_tile<BK, BV>(cur, kb, vb, knb, vnb, warp * kTileTok, g, t);
    for (int tl = warp; tl < ntl; tl += kDecWarps) {
      const int lt0 = tl * kTileTok;  // local token index of the tile
      if (tl + kDecWarps < ntl) load_tile<BK, BV>(nxt, kb, vb, knb, vnb, lt0 + kDecWarps * kTileTok, g, t);
      // ---------------- K side: S = K̂·Q (two independent MMA chains)
      float sa[NT][4], sb[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) sa[nt][e] = sb[nt][e] = 0.f;
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const uint32_t a0 = mykl[get_bits<2 * BK>(cur.k0, 4 * s * BK) << 5];
        const uint32_t a1 = mykl[get_bits<2 * BK>(cur.k1, 4 * s * BK) << 5];
        const uint32_t a2 = mykl[get_bits<2 * BK>(cur.k0, (4 * s + 2) * BK) << 5];
        const uint32_t a3 = mykl[get_bits<2 * BK>(cur.k1, (4 * s + 2) * BK) << 5];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          if (s & 1)
            mma16816(sb[nt], a0, a1, a2, a3, qf[s][nt].x, qf[s][nt].y);
          else
            mma16816(sa[nt], a0, a1, a2, a3, qf[s][nt].x, qf[s][nt].y);
        }
      }
      const bool v0 = tok0 + lt0 + g < p.seq, v1 = tok0 + lt0 + g + 8 < p.seq;
      // ---------------- online softmax per head h = 4nt + t (lanes of equal t)
      float w0[NT], w1[NT];  // p·s_v·fold for tokens g, g+8 of head 4nt+t
      bool need = false;
      float zz0[NT], zz1[NT], mx[NT];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        zz0[nt] = v0 ? (sa[nt][0] + sb[nt][0] + sa[nt][1] + sb[nt][1]) * cur.nk0 : -INFINITY;
        zz1[nt] = v1 ? (sa[nt][2] + sb[nt][2] + sa[nt][3] + sb[nt][3]) * cur.nk1 : -INFINITY;
        float m = fmaxf(zz0[nt], zz1[nt]);
        m = fmaxf(m, __shfl_xor_sync(kFull, m, 4));
        m = fmaxf(m, __shfl_xor_sync(kFull, m, 8));
        m = fmaxf(m, __shfl_xor_sync(kFull, m, 16));
        mx[nt] = m;
        need |= m > m_run[nt] + kLazy;
      }
      if (__any_sync(kFull, need)) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          if (mx[nt] > m_run[nt] + kLazy) {
            const float f = (m_run[nt] == -INFINITY) ? 0.f : ex2(m_run[nt] - mx[nt]);
            m_run[nt] = mx[nt];
            l_run[nt] *= f;
#pragma unroll
            for (int mt = 0; mt < 8; ++mt)
#pragma unroll
              for (int e = 0; e < 4; ++e) o[mt][nt][e] *= f;
          }
        }
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const float p0 = ex2(zz0[nt] - m_run[nt]);
        const float p1 = ex2(zz1[nt] - m_run[nt]);
        l_run[nt] += p0 + p1;
        w0[nt] = p0 * cur.nv0 * p.v_fold;
        w1[nt] = p1 * cur.nv1 * p.v_fold;
      }
      // ---------------- V side: B[k = token][n = col g] for tokens 2t,2t+1,2t+8,2t+9
      uint32_t bw[NT][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int h4 = (g >> 1);  // head within this n-tile (col g = 2·h4 + lo)
        const int src0 = 4 * (2 * t) + h4, src1 = 4 * (2 * t + 1) + h4;
        const float x0 = __shfl_sync(kFull, w0[nt], src0);  // token 2t
        const float x1 = __shfl_sync(kFull, w0[nt], src1);  // token 2t+1
        const float x2 = __shfl_sync(kFull, w1[nt], src0);  // token 2t+8
        const float x3 = __shfl_sync(kFull, w1[nt], src1);  // token 2t+9
        const bool head_ok = 4 * nt + h4 < G;
        float y0 = __half2float(__float2half_rn(x0)), y1 = __half2float(__float2half_rn(x1));
        float y2 = __half2float(__float2half_rn(x2)), y3 = __half2float(__float2half_rn(x3));
        if (g & 1) {  // lo column: the rounding residual of the hi column
          y0 = x0 - y0; y1 = x1 - y1; y2 = x2 - y2; y3 = x3 - y3;
        }
        bw[nt][0] = head_ok ? pack_f16x2(y0, y1) : 0u;
        bw[nt][1] = head_ok ? pack_f16x2(y2, y3) : 0u;
      }
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        // rows g / g+8 <-> coordinates 16g + 2mt / 16g + 2mt + 1
        const uint32_t a0 = myvl[get_bits<2 * BV>(cur.v0, (2 * mt) * 2 * BV) << 5];
        const uint32_t a1 = myvl[get_bits<2 * BV>(cur.v0, (2 * mt + 1) * 2 * BV) << 5];
        const uint32_t a2 = myvl[get_bits<2 * BV>(cur.v1, (2 * mt) * 2 * BV) << 5];
        const uint32_t a3 = myvl[get_bits<2 * BV>(cur.v1, (2 * mt + 1) * 2 * BV) << 5];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma16816(o[mt][nt], a0, a1, a2, a3, bw[nt][0], bw[nt][1]);
      }
      cur = nxt;
    }

    // ---------------- combine the 8 warps of the CTA, write the item's partials
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float l = l_run[nt];
      l += __shfl_xor_sync(kFull, l, 4);
      l += __shfl_xor_sync(kFull, l, 8);
      l += __shfl_xor_sync(kFull, l, 16);
      const int h = 4 * nt + t;
      if (h < G) {
        float* cw = comb + (warp * G + h) * 130;
        if (g == 0) {
          cw[0] = m_run[nt];
          cw[1] = l;
        }
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          cw[2 + 16 * g + 2 * mt] = o[mt][nt][0] + o[mt][nt][1];
          cw[2 + 16 * g + 2 * mt + 1] = o[mt][nt][2] + o[mt][nt][3];
        }
      }
    }
    __syncthreads();
    const int b = bk / p.Hkv, kvh = bk % p.Hkv;
    for (int e = tid; e < G * 128; e += blockDim.x) {
      const int h = e >> 7, dim = e & 127;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, comb[(w * G + h) * 130]);
      float L = 0.f, A = 0.f;
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) {
        const float mw = comb[(w * G + h) * 130];
        const float f = (mw == -INFINITY) ? 0.f : ex2(mw - M);
        L += f * comb[(w * G + h) * 130 + 1];
        A += f * comb[(w * G + h) * 130 + 2 + dim];
      }
      float* dst = p.part + (((size_t)b * p.Hq + kvh * G + h) * p.pl.S + sp) * 130;
      if (dim == 0) {
        dst[0] = M;
        dst[1] = L;
      }
      dst[2 + dim] = A;
    }
    __syncthreads();  // comb is reused by the next item
  }
}

// ------------------------------------------------------------------ merge
// One block (256 threads) per (batch, q head): log-sum-exp combine of the
// splits in the rotated domain, then out = Πᵀ·acc / L.  Π is staged in shared
// memory before the block waits for the split grid (programmatic launch), and
// the split loads are spread over the threads so they are in flight together.
__device__ __forceinline__ float block_reduce(float v, float* red, bool is_max) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float u = __shfl_xor_sync(kFull, v, o);
    v = is_max ? fmaxf(v, u) : v + u;
  }
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float r = red[0];
  for (int w = 1; w < (int)(blockDim.x >> 5); ++w) r = is_max ? fmaxf(r, red[w]) : r + red[w];
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(256) decode_merge_kernel(const float* __restrict__ pi,
                                                           const float* __restrict__ part, int S,
                                                           float* __restrict__ out) {
  extern __shared__ __align__(16) float msm[];
  float* spi = msm;               // Π, 128 x 128
  float* acc = spi + 128 * 128;   // [2][128]
  float* red = acc + 256;         // [8]
  float* w = red + 8;             // [S]
  const int tid = threadIdx.x, bh = blockIdx.x;
  {
    const float4* src = reinterpret_cast<const float4*>(pi);
    float4* dst = reinterpret_cast<float4*>(spi);
#pragma unroll
    for (int k = 0; k < 16; ++k) dst[tid + 256 * k] = __ldg(src + tid + 256 * k);
  }
  griddep_wait();  // partials of the split grid
  const float* P = part + (size_t)bh * S * 130;
  float mloc = -INFINITY;
  for (int s = tid; s < S; s += blockDim.x) {
    const float m = P[(size_t)s * 130];
    w[s] = m;
    mloc = fmaxf(mloc, m);
  }
  const float M = block_reduce(mloc, red, true);
  float lloc = 0.f;
  for (int s = tid; s < S; s += blockDim.x) {
    const float f = (w[s] == -INFINITY) ? 0.f : ex2(w[s] - M);
    lloc += f * P[(size_t)s * 130 + 1];
    w[s] = f;
  }
  const float L = block_reduce(lloc, red, false);  // its barriers also publish w[]
  const int i = tid & 127, hf = tid >> 7;
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
  int s = hf;
  for (; s + 6 < S; s += 8) {
    a0 += w[s] * P[(size_t)s * 130 + 2 + i];
    a1 += w[s + 2] * P[(size_t)(s + 2) * 130 + 2 + i];
    a2 += w[s + 4] * P[(size_t)(s + 4) * 130 + 2 + i];
    a3 += w[s + 6] * P[(size_t)(s + 6) * 130 + 2 + i];
  }
  for (; s < S; s += 2) a0 += w[s] * P[(size_t)s * 130 + 2 + i];
  acc[hf * 128 + i] = (a0 + a1) + (a2 + a3);
  __syncthreads();
  if (tid < 128) acc[i] += acc[128 + i];
  __syncthreads();
  // out_i = Σ_k Π[k][i] acc[k]: two halves of k, combined through shared memory
  float o = 0.f;
  const int k0 = hf * 64;
#pragma unroll 8
  for (int k = k0; k < k0 + 64; ++k) o = fmaf(spi[k * 128 + i], acc[k], o);
  if (hf == 1) acc[128 + i] = o;  // the loop above reads acc[0..127] only
  __syncthreads();
  if (hf == 0) out[(size_t)bh * 128 + i] = (o + acc[128 + i]) / L;
}

// cudaLaunchKernelEx with programmatic stream serialization: the grid may start
// while the previous grid in the stream finishes; it calls griddepcontrol.wait
// before touching anything that grid produces.
template <typename... Exp, typename... Act>
static cudaError_t launch_pdl(void (*kern)(Exp...), int grid, int block, size_t smem, cudaStream_t st,
                              Act&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Act>(args)...);
}

template <int BK, int BV, int G>
static cudaError_t run_split(const DecParams& p, cudaStream_t st) {
  auto k = decode_split_kernel<BK, BV, G>;
  static int attr_done = 0;  // the layout never exceeds 112 KB; set once, outside capture
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, 112 * 1024);
    if (e != cudaSuccess) return e;
    attr_done = 1;
  }
  const int items = p.B * p.Hkv * p.pl.S;
  const int grid = std::max(1, std::min(items, ctas_per_sm(G) * num_sms()));
  return launch_pdl(k, grid, 256, (size_t)p.sm.bytes, st, p);
}

template <int BK, int BV>
static cudaError_t run_split_g(const DecParams& p, cudaStream_t st) {
  switch (p.G) {
    case 1: return run_split<BK, BV, 1>(p, st);
    case 2: return run_split<BK, BV, 2>(p, st);
    case 4: return run_split<BK, BV, 4>(p, st);
    case 8: return run_split<BK, BV, 8>(p, st);
  }
  return cudaErrorInvalidValue;
}

template <int BK>
static cudaError_t run_split_v(const DecParams& p, int bv, cudaStream_t st) {
  switch (bv) {
    case 1: return run_split_g<BK, 1>(p, st);
    case 2: return run_split_g<BK, 2>(p, st);
    case 3: return run_split_g<BK, 3>(p, st);
    case 4: return run_split_g<BK, 4>(p, st);
  }
  return cudaErrorInvalidValue;
}

tq_status launch_decode(const DevCtx& kc, const DevCtx& vc, const void* q, int q_dtype,
                        const tq_codes* K, const tq_codes* V, int B, int Hq, int Hkv, int64_t seq,
                        int64_t cap, float scale, float* out, void* ws, size_t ws_bytes,
                        cudaStream_t stream) {
  if (cap % 16 != 0) return TQ_ERR_UNSUPPORTED;
  const int G = Hq / Hkv;
  bool same_lut = kc.b_mse == vc.b_mse && kc.alpha == vc.alpha;
  for (int k = 0; same_lut && k < (1 << kc.b_mse); ++k) same_lut = kc.cen[k] == vc.cen[k];
  const DecSmem sm = dec_smem(kc.b_mse, vc.b_mse, G, same_lut);
  const DecPlan pl = make_plan(B, Hq, Hkv, seq);
  uint2* frag = static_cast<uint2*>(ws);
  size_t frag_bytes = (size_t)B * Hkv * 8 * pl.NT * 32 * sizeof(uint2);
  float* part = reinterpret_cast<float*>(static_cast<char*>(ws) + (frag_bytes + 255) / 256 * 256);
  const float fold = scale * kLog2e / (kc.sqrt_d * kc.alpha);
  cudaError_t e = launch_pdl(decode_qprep_kernel, B * Hkv, 256, 0, stream, (const float*)kc.pi, q,
                             (int)(q_dtype == TQ_F16), Hq, G, pl.NT, fold, frag);
  if (e != cudaSuccess) return set_cuda_error(e);
  DecParams p;
  p.klut = kc.lut;
  p.vlut = vc.lut;
  p.v_fold = 1.f / (vc.alpha * vc.sqrt_d);
  p.kcodes = K->d_codes;
  p.knorm = K->d_norm;
  p.vcodes = V->d_codes;
  p.vnorm = V->d_norm;
  p.seq = seq;
  p.cap = cap;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = G;
  p.pl = pl;
  p.qfrag = frag;
  p.part = part;
  p.sm = sm;
  p.same_lut = same_lut ? 1 : 0;
  switch (kc.b_mse) {
    case 1: e = run_split_v<1>(p, vc.b_mse, stream); break;
    case 2: e = run_split_v<2>(p, vc.b_mse, stream); break;
    case 3: e = run_split_v<3>(p, vc.b_mse, stream); break;
    case 4: e = run_split_v<4>(p, vc.b_mse, stream); break;
    default: return TQ_ERR_UNSUPPORTED;
  }
  if (e != cudaSuccess) return set_cuda_error(e);
  const size_t msmem = (size_t)(128 * 128 + 256 + 8 + pl.S) * sizeof(float);
  static size_t merge_attr = 0;  // raised only when a larger split count needs it
  if (msmem > merge_attr) {
    e = cudaFuncSetAttribute(decode_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)std::max<size_t>(msmem, 80 * 1024));
    if (e != cudaSuccess) return set_cuda_error(e);
    merge_attr = std::max<size_t>(msmem, 80 * 1024);
  }
  e = launch_pdl(decode_merge_kernel, B * Hq, 256, msmem, stream, (const float*)vc.pi, (const float*)part,
                 pl.S, out);
  return e == cudaSuccess ? TQ_OK : set_cuda_error(e);
}

// ------------------------------------------------------------------ decode without a workspace
// Scratch for tq_decode_attention_noalloc: the query fragments and the split
// partials that tq_decode_attention keeps in the caller's workspace.  It is a
// file-scope device array, so the driver reserves it on every GPU that loads
// the library, and it stays reserved until the process exits.  Every call
// writes each byte of it that the call later reads, so nothing in it has to
// start at zero; concurrent calls (on different streams) would race on it.
constexpr size_t kNoAllocScratchBytes = (size_t)2 << 20;  // 2 MiB
static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

size_t decode_noalloc_limit() { return kNoAllocScratchBytes; }

// Device address of the scratch array on the current device.  The host-side
// symbol is only a stand-in, so the address is asked from the runtime once per
// device (with that device current) and cached.
static cudaError_t decode_scratch_address(void** out) {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = p;
  }
  *out = addr[dev];
  return cudaSuccess;
}

tq_status launch_decode_noalloc(const DevCtx& kc, const DevCtx& vc, const void* q, int q_dtype,
                                const tq_codes* K, const tq_codes* V, int B, int Hq, int Hkv,
                                int64_t seq, int64_t cap, float scale, float* out,
                                cudaStream_t stream) {
  const size_t need = decode_ws_bytes(kc.d, B, Hq, Hkv, seq);
  if (need > kNoAllocScratchBytes) return TQ_ERR_UNSUPPORTED;
  void* ws = nullptr;
  cudaError_t e = decode_scratch_address(&ws);
  if (e != cudaSuccess) return set_cuda_error(e);
  return launch_decode(kc, vc, q, q_dtype, K, V, B, Hq, Hkv, seq, cap, scale, out, ws, need, stream);
}

}  // namespace tq
