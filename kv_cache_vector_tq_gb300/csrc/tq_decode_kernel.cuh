#pragma once
// Decode attention over a TurboQuant_MSE KV cache (d = 128), one fused kernel
// per decode step.
//
// "TurboQuant 详解", section decode 阶段到底怎么“用”这些压缩后的 KV (second route):
// the kernel unpacks, looks up, scales and consumes the codes inside attention,
// never materialising fp16 K/V; and (same page, "decode 阶段") the token of the
// step is appended to the cache first.  "sub-byte-kv-cache-quantization-
// turboquant", section 工程实现的关键路径: the query is rotated once and query head
// h reads kv_head = h / (Hq / Hkv).
//
// Work split: S CTAs per (batch, KV head), each over a contiguous range of
// 16-token tiles; the grid fits the GPU in one wave (one CTA per SM).
//  1. Every CTA rotates the query heads of its KV head itself, q̂_h = Π·q_h,
//     with its slice of Π loaded before it waits for the previous grid (Π is
//     constant data), so the G·128·128 products cost no extra launch.
//  2. The CTA whose range holds position seq-1 also rotates the new K and V
//     (compensated dot products), encodes them (norm, bucketize against the
//     codebook thresholds, pack), writes them to the cache and patches them
//     into its staged tile; it takes half a share of the tiles to make room.
//  3. Every CTA streams its tiles: each lane copies its own 16-byte chunks
//     with cp.async into lane-private shared-memory slots, up to four tiles
//     ahead (a slot is refilled as soon as its tile's words are in registers),
//     and the warp runs
//       K side  S[t][n] = Σ_κ K̂[t][κ]·Q[κ][n]   (mma.m16n8k16: A from a pair
//               table indexed by two codes, B = pre-rotated queries, hi/lo)
//       softmax online per head in base 2 (scale folded into Q), lazy rescale
//       V side  O[μ][n] += Σ_t V̂[μ][t]·W[t][n]  (A from V pair blocks, which
//               hold two consecutive tokens' codes side by side; B = p·s_v)
//  4. The warps of a CTA merge their softmax states.  O stays in the rotated
//     domain up to here (Σ_t p_t s_t Πᵀŷ_t = Πᵀ Σ_t p_t s_t ŷ_t); the CTA applies
//     Πᵀ to its own partial, which commutes with the rescaled merge.
//  5. With S > 1 each CTA publishes (m, l, Πᵀ·acc) and the last CTA of the
//     (batch, KV head) to arrive merges the S partials into the output.
// TurboQuant_Prod keys (template flag Q; attention without an append, G <= 4):
// the logit gains the QJL term of the unbiased estimator ("TurboQuant 详解",
// section TurboQuant_prod), s·γ·√(π/2)/d·⟨S·q, 2·bits − 1⟩, as a second MMA
// chain per tile: A = ±1 pairs from a four-entry pair table indexed by two
// sign bits, B = S·q (rotated like q̂ from S in column slices, hi/lo, with the
// constants folded in); γ is staged with the tile's norms.
#include <algorithm>
#include <utility>

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {


constexpr int kTileTok = 16;
constexpr int kStages = 4;            // tiles in flight per warp
constexpr int kFieldBytes = 32 * 16;  // one 16-byte slot per lane
constexpr int kStageBytes = 4 * kFieldBytes + 128;  // + the tile's 16 K and 16 V norms
// Prod keys: + the tile's 16 γ (64 B) and its 16 tokens' sign words (4 each, 256 B)
constexpr int kQGamma = 4 * kFieldBytes + 128;
constexpr int kQSigns = kQGamma + 64;
constexpr int kStageBytesQ = kQSigns + 256;
__host__ __device__ constexpr int stage_bytes(bool q) { return q ? kStageBytesQ : kStageBytes; }
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLazy = 8.f;  // rescale only when the running max grows by > 2^8
constexpr int kPart = 132;    // floats per head in a published partial: m, l, 2 pad, acc[128]

// Workspace: one arrival counter per (batch, KV head), then the partial state
// (m, l, Πᵀ·acc[128]) of every CTA when a (batch, KV head) is split over more
// than one CTA.  Splits are only made while the grid fits one CTA per SM, so
// the number of partials is bounded by the SM count.
static size_t ws_counter_bytes(int groups) { return ((size_t)groups * 4 + 255) / 256 * 256; }

// ------------------------------------------------------------------ cp.async
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async8(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;\n" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }

template <int N>
__device__ __forceinline__ void copy_words(void* dst, const uint32_t* src) {
  if constexpr (N == 4) {
    cp_async16(dst, src);
  } else if constexpr (N == 2) {
    cp_async8(dst, src);
  } else {
#pragma unroll
    for (int i = 0; i < N; ++i) cp_async4(static_cast<uint32_t*>(dst) + i, src + i);
  }
}

// ------------------------------------------------------------------ small helpers
template <int N>
__device__ __forceinline__ void read_words(uint32_t (&w)[N], const unsigned char* src) {
  if constexpr (N == 4) {
    const uint4 v = *reinterpret_cast<const uint4*>(src);
    w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
  } else if constexpr (N == 2) {
    const uint2 v = *reinterpret_cast<const uint2*>(src);
    w[0] = v.x; w[1] = v.y;
  } else {
#pragma unroll
    for (int i = 0; i < N; ++i) w[i] = reinterpret_cast<const uint32_t*>(src)[i];
  }
}

__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = a + b;
  const float bb = s - a;
  e = (a - (s - bb)) + (b - bb);
}

// Read-only 16-byte load kept in program order with the grid-dependency wait
// (volatile), so that loads of constant data are in flight while it waits.
__device__ __forceinline__ float4 ldg_early(const float4* p) {
  float4 v;
  asm volatile("ld.global.nc.v4.f32 {%0, %1, %2, %3}, [%4];\n"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p));
  return v;
}


// ------------------------------------------------------------------ parameters
// Field order is part of the tuning: the fields the tile loop reads come first
// (inserting a pointer among them once cost ~0.3 us per call at b = 4).
struct StepParams {
  uint32_t* kcodes;
  float* knorm;
  uint32_t* vcodes;
  float* vnorm;
  int64_t seq, cap;
  const uint32_t* kqjl;   // Prod keys: sign words, 4 per token
  const float* krn;       // Prod keys: γ per token
  const float* vpi;       // Π of the V context, 128 x 128 row-major fp32 (output rotation)
  float vfold;  // 1 / (α_V·√d)
  float kfold;  // scale·log2(e) / (√d·α_K)
  float qfold;  // Prod keys: scale·log2(e)·√(π/2) / d (the QJL term)
  float sqrt_d;
  int B, Hq, Hkv, S, tiles;
  int same_lut;
  const float4* kslices;  // Π of the K context in column slices (see the rotation below)
  const float4* vslices;  // the same for the V context
  const uint32_t* klut;
  const uint32_t* vlut;
  const float4* sslices;  // Prod keys: S in column slices, like kslices
  int* status;    // device status word of the K context
  int* counters;  // [B*Hkv] arrival counters (zero between calls)
  float* part;    // [B*Hkv][S][G][kPart] per-CTA (m, l, Πᵀ·acc) when S > 1
  const void* q;
  const void* knew;
  const void* vnew;
  float* out;
  const uint32_t* klut_hi;  // b + 1/2 bits: the (b+1)-bit pair table (K and V share both tables)
  int q_f16;
  int new_f16;
  int append;
  float kthr[15];
  float vthr[15];
  int kv_shift;  // 1: Hkv counts virtual KV heads, two per cache head (vh >> 1)
};

// First tile of CTA u of the U CTAs that share a (batch, KV head).  With an
// appended token the last CTA, which owns position seq-1 and encodes the new
// K and V before it streams, takes half a share.
__host__ __device__ inline int split_begin(int u, int U, int tiles, bool append) {
  if (u >= U) return tiles;
  if (!append || U == 1) return (int)((int64_t)u * tiles / U);
  return (int)((int64_t)2 * u * tiles / (2 * U - 1));
}

// Shared-memory layout (bytes), computed identically on host and device.
// Each warp has kStages tile stages of four 512-byte fields (one 16-byte slot
// per lane: K codes of tokens g and g+8, V pair blocks t and t+4) and the
// tile's 16 K and 16 V norms,
// which after the tile loop hold its softmax state.
struct StepSmem {
  int vlut, qlut, stage, wreg, mw, qs, qhat, newin, ynew, newcodes, uni, opart, qfs, cpart, outp, flag, bytes;
};

// Offset in a warp region of its rows of Π_V: after its softmax state
// ((NT·512 + 16) floats) and its partial outputs (G·128 floats).
__host__ __device__ inline int pi_off(int G) {
  const int NT = (2 * G + 7) / 8, a = (NT * 512 + 16) * 4, b = G * 128 * 4;
  return ((a > b ? a : b) + 127) / 128 * 128;
}

__host__ __device__ inline StepSmem step_smem(int bk, int bv, int G, int W, bool same_lut, bool q,
                                             bool mx = false) {
  StepSmem m;
  const int NT = (2 * G + 7) / 8, NCH = W / 4;
  int o = (1 << (2 * bk)) * 32 * 4;
  m.vlut = o;  // b + 1/2 bits: where the (b+1)-bit table starts (V shares both tables)
  if (mx)
    o += (4 << (2 * bk)) * 32 * 4;
  else if (bk == 4 && bv == 4)
    o = 256 * 256;  // byte-indexed rows: K entries at lane·4, V entries at 128 + lane·4
  else if (!same_lut)
    o += (1 << (2 * bv)) * 32 * 4;
  m.qlut = o;  // Prod keys: the four ±1 sign pairs x32 lanes
  if (q) o += 4 * 32 * 4;
  o = (o + 127) / 128 * 128;
  // after the loop: its state (then its partial outputs), and its rows of Π_V at pi_off
  const int st = kStages * stage_bytes(q), cw = pi_off(G) + (128 / W) * 512;
  m.wreg = ((st > cw ? st : cw) + 127) / 128 * 128;
  m.stage = o;  // after the tile loop: the warps' states, then partial outputs [W][G][128]
  o += W * m.wreg;
  // [0, o) also holds the S published partials while the last CTA merges them
  m.mw = o;
  o += 16;
  m.qs = o;
  o += G * 128 * 4;  // the query heads in fp32
  m.qhat = o;
  o += G * 128 * 4;  // rotated queries
  m.newin = o;
  o += 2 * 128 * 4;  // k_new, v_new as fp32
  m.ynew = o;
  o += 2 * 128 * 4;  // rotated k_new, v_new
  m.newcodes = o;
  o += (16 + 32 + 32 + 4) * 4;  // K words, V slot bits, V slot mask, norms
  // one region used twice: the rotation's partial sums (and the appended
  // token's), then the query fragments, the warp-merged state and the output
  m.uni = o;
  m.opart = o + NCH * G * 128 * 4;
  m.qfs = o;
  m.cpart = o + 8 * NT * 32 * 8;
  m.outp = m.cpart + (NT * 512 + 16) * 4;
  const int u1 = NCH * G * 128 * 4 + NCH * 128 * 16, u2 = m.outp + G * 128 * 4 - o;
  o += u1 > u2 ? u1 : u2;
  m.flag = o;
  o += 16;
  m.bytes = (o + 127) / 128 * 128;
  return m;
}

// ------------------------------------------------------------------ the kernel
template <int BK, int BV, int G, int W, bool Q, bool MX = false, bool SH = false>
__global__ void __launch_bounds__(W * 32, 1) decode_step_kernel(const StepParams p) {
  constexpr int NT = (2 * G + 7) / 8;
  constexpr int WK = 4 * BK, WV = 4 * BV;  // words per vector
  constexpr int EK = 1 << (2 * BK), EV = 1 << (2 * BV);
  constexpr int NTH = W * 32;
  constexpr int NCH = W / 4;    // column chunks of the rotation (4 warps, 128 rows, per chunk)
  constexpr int CW = 128 / NCH;  // columns per chunk
  constexpr int NF4 = CW / 4;
  constexpr int RPW = 128 / W;  // Π_V rows per warp in the output rotation
  constexpr int QPT = (G * 128 + NTH - 1) / NTH;  // query elements per thread
  constexpr bool kByte = BK == 4 && BV == 4;      // pair codes are whole bytes
  static_assert(W % 4 == 0 && NTH >= 256, "4 warps per rotation chunk; a thread per new-token element");
  static_assert(!Q || (G <= 4 && BK <= 3), "Prod keys: up to 4 query heads per KV head, (b-1)-bit codes");
  // b + 1/2 bits per coordinate (MX): K and V both at b + 1/2 with the same
  // tables; coordinates j mod 16 < 8 take BK + 1 bits.  A vector is
  // WX = 2·(2·BK + 1) words; a lane's 32 K coordinates (or 16 V coordinate
  // pairs) are 16·(2·BK + 1) contiguous bits from a word or half-word boundary.
  static_assert(!MX || (!Q && BK == BV && BK <= 3), "b + 1/2 bits: MSE keys and values of equal b <= 3");
  constexpr int WX = 2 * (2 * BK + 1);
  constexpr int SB = stage_bytes(Q);
  extern __shared__ __align__(128) unsigned char smem[];
  const StepSmem L = step_smem(BK, BV, G, W, p.same_lut != 0, Q, MX);
  uint32_t* klut = reinterpret_cast<uint32_t*>(smem);
  uint32_t* khi = reinterpret_cast<uint32_t*>(smem + L.vlut);  // MX: the (BK+1)-bit table
  uint32_t* qlut = reinterpret_cast<uint32_t*>(smem + L.qlut);  // Prod keys
  uint32_t* vlut = (p.same_lut || MX) ? klut : reinterpret_cast<uint32_t*>(smem + L.vlut);
  unsigned char* stage = smem + L.stage;
  float* qs = reinterpret_cast<float*>(smem + L.qs);      // [G][128]
  float* qhat = reinterpret_cast<float*>(smem + L.qhat);  // [G][128]
  float* newin = reinterpret_cast<float*>(smem + L.newin);  // [2][128]
  float* ynew = reinterpret_cast<float*>(smem + L.ynew);    // [2][128]
  uint32_t* nk_words = reinterpret_cast<uint32_t*>(smem + L.newcodes);  // [16]
  uint32_t* nv_bits = nk_words + 16;                                     // [32]
  uint32_t* nv_mask = nv_bits + 32;                                      // [32]
  float* new_norm = reinterpret_cast<float*>(nv_mask + 32);              // [2]
  float* rpart = reinterpret_cast<float*>(smem + L.uni);     // [NCH][G][128]
  float4* opart = reinterpret_cast<float4*>(smem + L.opart);  // [NCH][128]
  uint2* qfs = reinterpret_cast<uint2*>(smem + L.qfs);       // [8][NT][32]
  float* cpart = reinterpret_cast<float*>(smem + L.cpart);   // [NT*512] fragment order, M[8], L[8]
  float* cM = cpart + NT * 512;
  float* cL = cM + 8;
  float* outp = reinterpret_cast<float*>(smem + L.outp);  // [G][128]
  int* flag = reinterpret_cast<int*>(smem + L.flag);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int grp = blockIdx.x / p.S, split = blockIdx.x % p.S;  // grp = b * Hkv + kvh
  const int b = grp / p.Hkv, kvh = grp % p.Hkv;
  const bool append = p.append != 0;
  const int t_begin = split_begin(split, p.S, p.tiles, append);
  const int t_end = split_begin(split + 1, p.S, p.tiles, append);
  const int ntl = t_end - t_begin;
  // SH (short loops: at most 8 tiles per warp, as in one decode layer of 16K
  // tokens): one tile in flight ahead of the one in use, so the first tiles
  // arrive sooner (12.56 against 12.80 us per call at b = 4).  Otherwise
  // kStages tiles in flight (a 128K-token layer: 66.7 against 67.7 us).  A
  // template choice: one loop holding both orders scheduled worse than either.
  constexpr bool shallow = SH;
  // vector index of token 0 of the group's cache head (virtual heads, plain
  // MSE caches only, share one; the others keep grp, which the register-bound
  // 3.5-bit kernel needs: 16.5 against 18.3 us per call with the shift)
  const int cgrp = (MX || Q) ? grp : b * (p.Hkv >> p.kv_shift) + (kvh >> p.kv_shift);
  const int64_t gbase = (int64_t)cgrp * p.cap;
  const int new_tile = (int)((p.seq - 1) / kTileTok), new_row = (int)((p.seq - 1) % kTileTok);
  const bool owner = append && new_tile >= t_begin && new_tile < t_end;
  unsigned char* my_stage = stage + warp * L.wreg;

  // ---- prologue on constant data (overlaps the previous grid where an SM is
  //      free): this thread's slice of Π_K (and, in the owner, of Π_V), the
  //      barriers, and the pair tables replicated per lane.  Thread (row, chunk)
  //      = (32(w%4) + lane, w/4) reads Π[row][chunk·CW ..+CW) from the slice
  //      table, where a warp's 32 rows of one slice column are contiguous.
  const int rrow = 32 * (warp & 3) + lane, rc0 = (warp >> 2) * CW;
  float4 pk[NF4], pv[NF4];
#pragma unroll
  for (int j = 0; j < NF4; ++j) {
    const int col = rc0 + 4 * j;
    pk[j] = ldg_early(p.kslices + ((col >> 5) * 8 + ((col & 31) >> 2)) * 128 + rrow);
  }
  if (owner) {
#pragma unroll
    for (int j = 0; j < NF4; ++j) {
      const int col = rc0 + 4 * j;
      pv[j] = ldg_early(p.vslices + ((col >> 5) * 8 + ((col & 31) >> 2)) * 128 + rrow);
    }
  }
  float4 ps[Q ? NF4 : 1];  // Prod keys: this thread's slice of S
  if constexpr (Q) {
#pragma unroll
    for (int j = 0; j < NF4; ++j) {
      const int col = rc0 + 4 * j;
      ps[j] = ldg_early(p.sslices + ((col >> 5) * 8 + ((col & 31) >> 2)) * 128 + rrow);
    }
    // sign pair table: entry i = (2·(i & 1) − 1, 2·(i >> 1) − 1) in fp16, x32 lanes
    for (int i = tid; i < 4 * 32; i += NTH) {
      const uint32_t e = (uint32_t)(i >> 5);
      qlut[i] = ((e & 1u) ? 0x3C00u : 0xBC00u) | ((e & 2u) ? 0x3C000000u : 0xBC000000u);
    }
  }
  for (int i = tid; i < 16 + 32 + 32; i += NTH) nk_words[i] = 0u;
  if constexpr (kByte) {  // row i: K entry x32 lanes, then V entry x32 lanes
    constexpr int NB = 256 * 16 / NTH;
    uint32_t v[NB];
#pragma unroll
    for (int k = 0; k < NB; ++k) {
      const int i = tid + k * NTH;
      v[k] = __ldg(((i >> 3) & 1 ? p.vlut : p.klut) + (i >> 4));
    }
#pragma unroll
    for (int k = 0; k < NB; ++k) reinterpret_cast<uint4*>(smem)[tid + k * NTH] = make_uint4(v[k], v[k], v[k], v[k]);
  } else {
    constexpr int NK = (EK * 8 + NTH - 1) / NTH;
    uint32_t v[NK];
#pragma unroll
    for (int k = 0; k < NK; ++k) {
      const int i = tid + k * NTH;
      v[k] = i < EK * 8 ? __ldg(p.klut + (i >> 3)) : 0u;
    }
#pragma unroll
    for (int k = 0; k < NK; ++k) {
      const int i = tid + k * NTH;
      if (i < EK * 8) reinterpret_cast<uint4*>(klut)[i] = make_uint4(v[k], v[k], v[k], v[k]);
    }
    if constexpr (MX) {  // the (BK+1)-bit table, 4·EK entries
      constexpr int NH = (4 * EK * 8 + NTH - 1) / NTH;
      uint32_t u[NH];
#pragma unroll
      for (int k = 0; k < NH; ++k) {
        const int i = tid + k * NTH;
        u[k] = i < 4 * EK * 8 ? __ldg(p.klut_hi + (i >> 3)) : 0u;
      }
#pragma unroll
      for (int k = 0; k < NH; ++k) {
        const int i = tid + k * NTH;
        if (i < 4 * EK * 8) reinterpret_cast<uint4*>(khi)[i] = make_uint4(u[k], u[k], u[k], u[k]);
      }
    } else if (!p.same_lut) {
      constexpr int NV = (EV * 8 + NTH - 1) / NTH;
      uint32_t u[NV];
#pragma unroll
      for (int k = 0; k < NV; ++k) {
        const int i = tid + k * NTH;
        u[k] = i < EV * 8 ? __ldg(p.vlut + (i >> 3)) : 0u;
      }
#pragma unroll
      for (int k = 0; k < NV; ++k) {
        const int i = tid + k * NTH;
        if (i < EV * 8) reinterpret_cast<uint4*>(vlut)[i] = make_uint4(u[k], u[k], u[k], u[k]);
      }
    }
  }
  __syncthreads();
  griddep_wait();    // the cache, q and the new token may come from earlier grids
  griddep_launch();  // the next grid may start its own prologue as SMs free up

  // ---- inputs of the step, requested before the tile copies queue up
  float qv[QPT];
#pragma unroll
  for (int k = 0; k < QPT; ++k) {
    const int e = tid + k * NTH;
    qv[k] = 0.f;
    if (e < G * 128) {
      const int64_t off = ((int64_t)b * p.Hq + kvh * G + (e >> 7)) * 128 + (e & 127);
      qv[k] = p.q_f16 ? __half2float(static_cast<const __half*>(p.q)[off]) : static_cast<const float*>(p.q)[off];
    }
  }
  float nv = 0.f;  // owner: element tid of [k_new; v_new]
  if (owner && tid < 256) {
    const void* src = tid >= 128 ? p.vnew : p.knew;
    const int64_t off = (int64_t)cgrp * 128 + (tid & 127);
    nv = p.new_f16 ? __half2float(static_cast<const __half*>(src)[off]) : static_cast<const float*>(src)[off];
  }
  auto issue = [&](int j) {  // warp-local tile j -> stage j % kStages, one 16-byte slot per lane
    const int tile = t_begin + warp + j * W;
    if (tile < t_end) {
      unsigned char* st = my_stage + (j % kStages) * SB;
      const int64_t vb = gbase + (int64_t)tile * kTileTok;
      if constexpr (MX) {
        // BK + 1 words from the word holding the lane's first bit (bit
        // 16·(2·BK + 1)·t of a K row, ·g of a V pair block)
        const int ko = (t * (2 * BK + 1)) >> 1, vo = (g * (2 * BK + 1)) >> 1;
        if constexpr (BK == 2) {
          // 2.5 bits: four words from the even (8-byte aligned) word at or
          // below the first, in two 8-byte copies (rows of 10 words, pair
          // blocks of 20: every lane's four words stay inside its row/block)
          const int ke = ko & ~1, ve = vo & ~1;
#pragma unroll
          for (int w = 0; w < 2; ++w) {
            cp_async8(st + 0 * kFieldBytes + lane * 16 + 8 * w, p.kcodes + (vb + g) * WX + ke + 2 * w);
            cp_async8(st + 1 * kFieldBytes + lane * 16 + 8 * w, p.kcodes + (vb + g + 8) * WX + ke + 2 * w);
            cp_async8(st + 2 * kFieldBytes + lane * 16 + 8 * w, p.vcodes + (vb + 2 * t) * WX + ve + 2 * w);
            cp_async8(st + 3 * kFieldBytes + lane * 16 + 8 * w, p.vcodes + (vb + 2 * t + 8) * WX + ve + 2 * w);
          }
        } else {
#pragma unroll
          for (int w = 0; w <= BK; ++w) {
            cp_async4(st + 0 * kFieldBytes + lane * 16 + 4 * w, p.kcodes + (vb + g) * WX + ko + w);
            cp_async4(st + 1 * kFieldBytes + lane * 16 + 4 * w, p.kcodes + (vb + g + 8) * WX + ko + w);
            cp_async4(st + 2 * kFieldBytes + lane * 16 + 4 * w, p.vcodes + (vb + 2 * t) * WX + vo + w);
            cp_async4(st + 3 * kFieldBytes + lane * 16 + 4 * w, p.vcodes + (vb + 2 * t + 8) * WX + vo + w);
          }
        }
      } else {
        copy_words<BK>(st + 0 * kFieldBytes + lane * 16, p.kcodes + (vb + g) * WK + t * BK);
        copy_words<BK>(st + 1 * kFieldBytes + lane * 16, p.kcodes + (vb + g + 8) * WK + t * BK);
        // V pair blocks t and t+4 of the tile; this lane's coordinates 16g..16g+15
        copy_words<BV>(st + 2 * kFieldBytes + lane * 16, p.vcodes + (vb + 2 * t) * WV + g * BV);
        copy_words<BV>(st + 3 * kFieldBytes + lane * 16, p.vcodes + (vb + 2 * t + 8) * WV + g * BV);
      }
      if (lane < 8)  // lanes 0-3: the 16 K norms, lanes 4-7: the 16 V norms
        cp_async16(st + 4 * kFieldBytes + lane * 16, (lane < 4 ? p.knorm : p.vnorm) + vb + 4 * (lane & 3));
      if constexpr (Q) {  // lanes 8-11: the 16 γ; lanes 12-27: the 16 tokens' sign words
        if (lane >= 8 && lane < 12) cp_async16(st + kQGamma + (lane - 8) * 16, p.krn + vb + 4 * (lane - 8));
        if (lane >= 12 && lane < 28) cp_async16(st + kQSigns + (lane - 12) * 16, p.kqjl + (vb + lane - 12) * 4);
      }
    }
    cp_async_commit();  // always, so that the group count stays uniform
  };
  issue(0);  // one tile per warp now; the rest after the rotation, which would queue behind them
#pragma unroll
  for (int k = 0; k < QPT; ++k)
    if (tid + k * NTH < G * 128) qs[tid + k * NTH] = qv[k];
  if (owner && tid < 256) newin[tid] = nv;
  __syncthreads();

  // ---- 1. q̂_h = Π_K·q_h: thread (row, chunk) sums over its chunk's columns
  //         (all lanes read the same query words), the chunks meet in rpart
  {
    float acc[G];
#pragma unroll
    for (int h = 0; h < G; ++h) acc[h] = 0.f;
#pragma unroll
    for (int j = 0; j < NF4; ++j) {
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float4 x = *reinterpret_cast<const float4*>(qs + h * 128 + rc0 + 4 * j);
        acc[h] = fmaf(pk[j].x, x.x, fmaf(pk[j].y, x.y, fmaf(pk[j].z, x.z, fmaf(pk[j].w, x.w, acc[h]))));
      }
    }
#pragma unroll
    for (int h = 0; h < G; ++h) rpart[((warp >> 2) * G + h) * 128 + rrow] = acc[h];
    if constexpr (Q) {  // S·q_h the same way; partial sums where the owner's would go
      float* spart = reinterpret_cast<float*>(opart);
#pragma unroll
      for (int h = 0; h < G; ++h) acc[h] = 0.f;
#pragma unroll
      for (int j = 0; j < NF4; ++j) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float4 x = *reinterpret_cast<const float4*>(qs + h * 128 + rc0 + 4 * j);
          acc[h] = fmaf(ps[j].x, x.x, fmaf(ps[j].y, x.y, fmaf(ps[j].z, x.z, fmaf(ps[j].w, x.w, acc[h]))));
        }
      }
#pragma unroll
      for (int h = 0; h < G; ++h) spart[((warp >> 2) * G + h) * 128 + rrow] = acc[h];
    }
  }
  if (owner) {
    // ---- 2a. the appended token, rotated as a compensated dot product
    //          (products split exactly with an FMA, sums by error-free
    //          two-sums) so that its codes agree with the encoder's up to
    //          coordinates within ~1e-6 of a codebook threshold
    auto dot2 = [&](const float4 (&pr)[NF4], const float* x, float& hi, float& lo) {
      hi = 0.f;
      lo = 0.f;
#pragma unroll
      for (int j = 0; j < NF4; ++j) {
        const float4 xv = *reinterpret_cast<const float4*>(x + rc0 + 4 * j);
        const float pa[4] = {pr[j].x, pr[j].y, pr[j].z, pr[j].w}, xa[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float pp = pa[e] * xa[e];
          const float er = fmaf(pa[e], xa[e], -pp);
          float s, err;
          two_sum(hi, pp, s, err);
          hi = s;
          lo += err + er;
        }
      }
    };
    float kh, kl, vh, vl;
    dot2(pk, newin, kh, kl);
    dot2(pv, newin + 128, vh, vl);
    opart[(warp >> 2) * 128 + rrow] = make_float4(kh, kl, vh, vl);
  }
  __syncthreads();
  for (int e = tid; e < G * 128; e += NTH) {  // sum the column chunks
    const int h = e >> 7, row = e & 127;
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < NCH; ++c) s += rpart[(c * G + h) * 128 + row];
    qhat[e] = s;
    if constexpr (Q) {  // S·q_h into the (unused) new-token buffers
      const float* spart = reinterpret_cast<const float*>(opart);
      float u = 0.f;
#pragma unroll
      for (int c = 0; c < NCH; ++c) u += spart[(c * G + h) * 128 + row];
      newin[e] = u;
    }
  }
  if (owner) {
    // ---- 2b. encode the appended K and V: norm, bucketize, pack, store
    if (tid < 256) {
      const int which = tid >> 7, row = tid & 127;
      float hi = 0.f, lo = 0.f;
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
        const float4 v = opart[c * 128 + row];
        float s, err;
        two_sum(hi, which ? v.z : v.x, s, err);
        hi = s;
        lo += (which ? v.w : v.y) + err;
      }
      ynew[tid] = hi + lo;
    }
    if (tid < 64) {  // norms (warp 0: K, warp 1: V), each lane 4 squares, then a tree
      const int which = tid >> 5;
      float ss = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float x = newin[which * 128 + lane + 32 * i];
        ss = fmaf(x, x, ss);
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(kFull, ss, off);
      if (lane == 0) new_norm[which] = sqrtf(ss);
    }
    __syncthreads();
    // unit-variance coordinate √d·y/‖x‖ against the codebook thresholds
    const int slot = (int)((p.seq - 1) & 1);
    if (tid < 256) {
      const int which = tid >> 7, i = tid & 127;
      const float s = new_norm[which];
      uint32_t code = 0;
      if (s > 0.f) {
        const float v = ynew[tid] * (p.sqrt_d / s);
        const int nb = which ? BV : BK;
        const float* thr = which ? p.vthr : p.kthr;
        for (int k = 0; k < (1 << nb) - 1; ++k) code += v >= thr[k] ? 1u : 0u;
      }
      if (which == 0) {
        const int pos = i * BK;
        atomicOr(&nk_words[pos >> 5], code << (pos & 31));
        if ((pos & 31) + BK > 32) atomicOr(&nk_words[(pos >> 5) + 1], code >> (32 - (pos & 31)));
      } else {
        const int pos = (2 * i + slot) * BV;
        const uint32_t m = (1u << BV) - 1u;
        atomicOr(&nv_bits[pos >> 5], code << (pos & 31));
        atomicOr(&nv_mask[pos >> 5], m << (pos & 31));
        if ((pos & 31) + BV > 32) {
          atomicOr(&nv_bits[(pos >> 5) + 1], code >> (32 - (pos & 31)));
          atomicOr(&nv_mask[(pos >> 5) + 1], m >> (32 - (pos & 31)));
        }
      }
    }
    __syncthreads();
    const int64_t pos = gbase + p.seq - 1;
    if (tid < WK) p.kcodes[pos * WK + tid] = nk_words[tid];
    if (tid < 2 * WV) {
      uint32_t* w = p.vcodes + (pos >> 1) * (2 * WV) + tid;
      atomicAnd(w, ~nv_mask[tid]);
      atomicOr(w, nv_bits[tid]);
    }
    if (tid == 0) {
      p.knorm[pos] = new_norm[0];
      p.vnorm[pos] = new_norm[1];
    }
  }
  __syncthreads();

  // ---- query B fragments, built once for all warps: b0 = (K index 16s+2t.., col g),
  //      b1 = (16s+8+2t.., col g); K index 16s+8h+2t+e <-> coordinate 32t+4s+2h+e;
  //      col n = 2·head + (1 for the fp16 rounding residual).  The merged state
  //      beside them starts at zero.
  for (int e = tid; e < 8 * NT * 32; e += NTH) {
    const int ln = e & 31, nt = (e >> 5) % NT, s8 = (e >> 5) / NT;
    const int n = nt * 8 + (ln >> 2), h = n >> 1;
    uint2 f = make_uint2(0u, 0u);
    if (h < G) {
      const float4 x = *reinterpret_cast<const float4*>(qhat + h * 128 + 32 * (ln & 3) + 4 * s8);
      uint32_t h0, l0, h1, l1;
      split2(x.x * p.kfold, x.y * p.kfold, h0, l0);
      split2(x.z * p.kfold, x.w * p.kfold, h1, l1);
      f = (n & 1) ? make_uint2(l0, l1) : make_uint2(h0, h1);
    }
    qfs[e] = f;
    if constexpr (Q) {  // the same fragments of qfold·S·q_h, where the merged state goes later
      uint2 fq = make_uint2(0u, 0u);
      if (h < G) {
        const float4 x = *reinterpret_cast<const float4*>(newin + h * 128 + 32 * (ln & 3) + 4 * s8);
        uint32_t h0, l0, h1, l1;
        split2(x.x * p.qfold, x.y * p.qfold, h0, l0);
        split2(x.z * p.qfold, x.w * p.qfold, h1, l1);
        fq = (n & 1) ? make_uint2(l0, l1) : make_uint2(h0, h1);
      }
      reinterpret_cast<uint2*>(cpart)[e] = fq;
    }
  }
  __syncthreads();
  uint2 qf[8][NT];
  uint2 qsf[Q ? 8 : 1][NT];
#pragma unroll
  for (int s = 0; s < 8; ++s)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      qf[s][nt] = qfs[(s * NT + nt) * 32 + lane];
      if constexpr (Q) qsf[s][nt] = reinterpret_cast<const uint2*>(cpart)[(s * NT + nt) * 32 + lane];
    }
  if constexpr (!shallow) {
#pragma unroll
    for (int j = 1; j < kStages; ++j) issue(j);
  }

  // ---- 3. stream the tiles
  const uint32_t* mykl = klut + lane;
  const uint32_t* mykh = khi + lane;  // MX: the (BK+1)-bit table
  const uint32_t* myvl = vlut + lane;
  const uint32_t lane4 = lane * 4;
  const uint32_t tbase = smem_u32(smem);  // shared-window address of the byte-row tables
  float m_run[NT], l_run[NT];
  float o[8][NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    m_run[nt] = -INFINITY;
    l_run[nt] = 0.f;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) o[mt][nt][0] = o[mt][nt][1] = o[mt][nt][2] = o[mt][nt][3] = 0.f;
  }
  // this warp's rows of Π_V for the output rotation, copied into its own region
  // (asynchronous: nothing waits on them before the rotation at the end)
  auto issue_pv = [&]() {
    float* prow = reinterpret_cast<float*>(my_stage + pi_off(G));
#pragma unroll
    for (int r = 0; r < RPW; ++r) cp_async16(prow + r * 128 + 4 * lane, p.vpi + (warp * RPW + r) * 128 + 4 * lane);
    cp_async_commit();
  };
  // issued in the warp's last tile when it has one (Prod keys: after the loop)
  const bool pv_in_loop = warp < ntl;
  for (int j = 0; warp + j * W < ntl; ++j) {
    const int tile = t_begin + warp + j * W;
    if constexpr (shallow) {  // the next tile into another stage, then this one complete
      issue(j + 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<kStages - 1>();
    }
    const unsigned char* st = my_stage + (j % kStages) * SB;
    constexpr int KN = MX ? BK + 1 : BK, VN = MX ? BV + 1 : BV;
    uint32_t k0[KN], k1[KN], v0w[VN], v1w[VN];
    if constexpr (MX && BK == 2) {  // drop the leading word where the first one was odd
      uint32_t a[4], b2[4], c[4], d[4];
      read_words<4>(a, st + 0 * kFieldBytes + lane * 16);
      read_words<4>(b2, st + 1 * kFieldBytes + lane * 16);
      read_words<4>(c, st + 2 * kFieldBytes + lane * 16);
      read_words<4>(d, st + 3 * kFieldBytes + lane * 16);
      const bool kodd = ((t * 5) >> 1) & 1, vodd = ((g * 5) >> 1) & 1;
#pragma unroll
      for (int w = 0; w < 3; ++w) {
        k0[w] = kodd ? a[w + 1] : a[w];
        k1[w] = kodd ? b2[w + 1] : b2[w];
        v0w[w] = vodd ? c[w + 1] : c[w];
        v1w[w] = vodd ? d[w + 1] : d[w];
      }
    } else {
      read_words<KN>(k0, st + 0 * kFieldBytes + lane * 16);
      read_words<KN>(k1, st + 1 * kFieldBytes + lane * 16);
      read_words<VN>(v0w, st + 2 * kFieldBytes + lane * 16);
      read_words<VN>(v1w, st + 3 * kFieldBytes + lane * 16);
    }
    if constexpr (MX) {  // bring the lane's first bit to bit 0 (odd t for K, odd g for V)
      const uint32_t ks = (uint32_t)(t & 1) * 16u, vs = (uint32_t)(g & 1) * 16u;
#pragma unroll
      for (int w = 0; w + 1 < KN; ++w) {
        k0[w] = __funnelshift_r(k0[w], k0[w + 1], ks);
        k1[w] = __funnelshift_r(k1[w], k1[w + 1], ks);
        v0w[w] = __funnelshift_r(v0w[w], v0w[w + 1], vs);
        v1w[w] = __funnelshift_r(v1w[w], v1w[w + 1], vs);
      }
      k0[KN - 1] >>= ks;
      k1[KN - 1] >>= ks;
      v0w[VN - 1] >>= vs;
      v1w[VN - 1] >>= vs;
    }
    const float* ns = reinterpret_cast<const float*>(st + 4 * kFieldBytes);
    float4 nrm = make_float4(ns[g], ns[g + 8], ns[16 + g], ns[16 + g + 8]);
    // Prod keys: this tile's sign words (bits j = 32t + 4s + {0..3} of tokens g,
    // g+8) and γ, read before the stage is refilled below
    uint32_t qw0 = 0u, qw1 = 0u;
    float gam0 = 0.f, gam1 = 0.f;
    if constexpr (Q) {
      const uint32_t* sw = reinterpret_cast<const uint32_t*>(st + kQSigns);
      qw0 = sw[g * 4 + t];
      qw1 = sw[(g + 8) * 4 + t];
      const float* gm = reinterpret_cast<const float*>(st + kQGamma);
      gam0 = gm[g];
      gam1 = gm[g + 8];
    }
    if (!MX && owner && tile == new_tile) {  // the appended token: use the codes just made
      if (new_row == g) {
#pragma unroll
        for (int w = 0; w < BK; ++w) k0[w] = nk_words[t * BK + w];
        nrm.x = new_norm[0];
        nrm.z = new_norm[1];
      }
      if (new_row == g + 8) {
#pragma unroll
        for (int w = 0; w < BK; ++w) k1[w] = nk_words[t * BK + w];
        nrm.y = new_norm[0];
        nrm.w = new_norm[1];
      }
      const int pbn = new_row >> 1;
      if ((pbn & 3) == t) {
#pragma unroll
        for (int w = 0; w < BV; ++w) {
          const uint32_t m = nv_mask[g * BV + w], nb = nv_bits[g * BV + w];
          if (pbn < 4)
            v0w[w] = (v0w[w] & ~m) | nb;
          else
            v1w[w] = (v1w[w] & ~m) | nb;
        }
      }
    }
    // every lane's words are in registers: refill this stage
    if constexpr (!shallow) issue(j + kStages);
    if (warp + (j + 1) * W >= ntl) issue_pv();  // the warp's last tile: its region is free now
    const int lt0 = tile * kTileTok;
    // K side: S = K̂·Q with two independent MMA chains
    float sa[NT][4], sb[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) sa[nt][e] = sb[nt][e] = 0.f;
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      uint32_t a0, a1, a2, a3;
      if constexpr (kByte) {  // a0/a2: bytes 2(s&1), 2(s&1)+1 of word s/2 (a1/a3 likewise from k1)
        a0 = lds_at<0>(tbase + byte_row_addr(k0[s >> 1], lane4, 2 * (s & 1)));
        a1 = lds_at<0>(tbase + byte_row_addr(k1[s >> 1], lane4, 2 * (s & 1)));
        a2 = lds_at<0>(tbase + byte_row_addr(k0[s >> 1], lane4, 2 * (s & 1) + 1));
        a3 = lds_at<0>(tbase + byte_row_addr(k1[s >> 1], lane4, 2 * (s & 1) + 1));
      } else if constexpr (MX) {  // coordinates 4s..4s+3 of the lane's 32: BK + 1 bits for s mod 4 < 2
        const int p0 = mixed_pos(4 * s, BK), p2 = mixed_pos(4 * s + 2, BK);
        if ((s & 2) == 0) {
          a0 = mykh[get_bits<2 * BK + 2>(k0, p0) << 5];
          a1 = mykh[get_bits<2 * BK + 2>(k1, p0) << 5];
          a2 = mykh[get_bits<2 * BK + 2>(k0, p2) << 5];
          a3 = mykh[get_bits<2 * BK + 2>(k1, p2) << 5];
        } else {
          a0 = mykl[get_bits<2 * BK>(k0, p0) << 5];
          a1 = mykl[get_bits<2 * BK>(k1, p0) << 5];
          a2 = mykl[get_bits<2 * BK>(k0, p2) << 5];
          a3 = mykl[get_bits<2 * BK>(k1, p2) << 5];
        }
      } else {
        a0 = mykl[get_bits<2 * BK>(k0, 4 * s * BK) << 5];
        a1 = mykl[get_bits<2 * BK>(k1, 4 * s * BK) << 5];
        a2 = mykl[get_bits<2 * BK>(k0, (4 * s + 2) * BK) << 5];
        a3 = mykl[get_bits<2 * BK>(k1, (4 * s + 2) * BK) << 5];
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        if (s & 1)
          mma16816(sb[nt], a0, a1, a2, a3, qf[s][nt].x, qf[s][nt].y);
        else
          mma16816(sa[nt], a0, a1, a2, a3, qf[s][nt].x, qf[s][nt].y);
      }
    }
    // Prod keys: Σ_j (S·q)_j·(2·bit_j − 1) for tokens g, g+8, sign bits j = 32t + 4s + {0..3}
    float qa[NT][4], qb[NT][4];
    if constexpr (Q) {
      const uint32_t w0 = qw0, w1 = qw1;
      const uint32_t* myql = qlut + lane;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) qa[nt][e] = qb[nt][e] = 0.f;
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const uint32_t a0 = myql[((w0 >> (4 * s)) & 3u) << 5];
        const uint32_t a1 = myql[((w1 >> (4 * s)) & 3u) << 5];
        const uint32_t a2 = myql[((w0 >> (4 * s + 2)) & 3u) << 5];
        const uint32_t a3 = myql[((w1 >> (4 * s + 2)) & 3u) << 5];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          if (s & 1)
            mma16816(qb[nt], a0, a1, a2, a3, qsf[s][nt].x, qsf[s][nt].y);
          else
            mma16816(qa[nt], a0, a1, a2, a3, qsf[s][nt].x, qsf[s][nt].y);
        }
      }
    }
    const bool ok0 = lt0 + g < p.seq, ok1 = lt0 + g + 8 < p.seq;
    // online softmax per head h = 4nt + t (lanes of equal t share a head)
    float w0[NT], w1[NT];
    bool need = false;
    float zz0[NT], zz1[NT], mx[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float z0 = sa[nt][0] + sb[nt][0] + sa[nt][1] + sb[nt][1];
      float z1 = sa[nt][2] + sb[nt][2] + sa[nt][3] + sb[nt][3];
      if constexpr (Q) {
        z0 = fmaf(gam0, qa[nt][0] + qb[nt][0] + qa[nt][1] + qb[nt][1], z0);
        z1 = fmaf(gam1, qa[nt][2] + qb[nt][2] + qa[nt][3] + qb[nt][3], z1);
      }
      zz0[nt] = ok0 ? z0 * nrm.x : -INFINITY;
      zz1[nt] = ok1 ? z1 * nrm.y : -INFINITY;
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
      w0[nt] = p0 * nrm.z * p.vfold;
      w1[nt] = p1 * nrm.w * p.vfold;
    }
    // V side: B[k = token][n = col g] for tokens 2t, 2t+1, 2t+8, 2t+9
    uint32_t bw[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int h4 = g >> 1;  // head within this n-tile (col g = 2·h4 + lo)
      const int src0 = 4 * (2 * t) + h4, src1 = 4 * (2 * t + 1) + h4;
      const float x0 = __shfl_sync(kFull, w0[nt], src0);
      const float x1 = __shfl_sync(kFull, w0[nt], src1);
      const float x2 = __shfl_sync(kFull, w1[nt], src0);
      const float x3 = __shfl_sync(kFull, w1[nt], src1);
      uint32_t h0, l0, h1, l1;
      split2(x0, x1, h0, l0);
      split2(x2, x3, h1, l1);
      const bool head_ok = 4 * nt + h4 < G;
      bw[nt][0] = head_ok ? ((g & 1) ? l0 : h0) : 0u;  // odd columns: the rounding residual
      bw[nt][1] = head_ok ? ((g & 1) ? l1 : h1) : 0u;
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      // rows g / g+8 <-> coordinates 16g + 2mt / 16g + 2mt + 1
      uint32_t a0, a1, a2, a3;
      if constexpr (kByte) {  // bytes 2(mt&1), 2(mt&1)+1 of word mt/2
        a0 = lds_at<128>(tbase + byte_row_addr(v0w[mt >> 1], lane4, 2 * (mt & 1)));
        a1 = lds_at<128>(tbase + byte_row_addr(v0w[mt >> 1], lane4, 2 * (mt & 1) + 1));
        a2 = lds_at<128>(tbase + byte_row_addr(v1w[mt >> 1], lane4, 2 * (mt & 1)));
        a3 = lds_at<128>(tbase + byte_row_addr(v1w[mt >> 1], lane4, 2 * (mt & 1) + 1));
      } else if constexpr (MX) {  // pair fields of coordinates 2mt, 2mt+1: BV + 1 bits each for mt < 4
        const int q0 = 2 * mixed_pos(2 * mt, BV), q1 = 2 * mixed_pos(2 * mt + 1, BV);
        if (mt < 4) {
          a0 = mykh[get_bits<2 * BV + 2>(v0w, q0) << 5];
          a1 = mykh[get_bits<2 * BV + 2>(v0w, q1) << 5];
          a2 = mykh[get_bits<2 * BV + 2>(v1w, q0) << 5];
          a3 = mykh[get_bits<2 * BV + 2>(v1w, q1) << 5];
        } else {
          a0 = myvl[get_bits<2 * BV>(v0w, q0) << 5];
          a1 = myvl[get_bits<2 * BV>(v0w, q1) << 5];
          a2 = myvl[get_bits<2 * BV>(v1w, q0) << 5];
          a3 = myvl[get_bits<2 * BV>(v1w, q1) << 5];
        }
      } else {
        a0 = myvl[get_bits<2 * BV>(v0w, (2 * mt) * 2 * BV) << 5];
        a1 = myvl[get_bits<2 * BV>(v0w, (2 * mt + 1) * 2 * BV) << 5];
        a2 = myvl[get_bits<2 * BV>(v1w, (2 * mt) * 2 * BV) << 5];
        a3 = myvl[get_bits<2 * BV>(v1w, (2 * mt + 1) * 2 * BV) << 5];
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) mma16816(o[mt][nt], a0, a1, a2, a3, bw[nt][0], bw[nt][1]);
    }
  }
  if (pv_in_loop) {
    cp_async_wait<1>();  // every tile copy is done; the Π_V rows may still be in flight
  } else {
    cp_async_wait_all();
    issue_pv();
  }

  // ---- 4. merge the warps and rotate back.  Each warp leaves its state in its
  //         own region in fragment order: acc value (nt, mt, e) of lane l at
  //         ((nt·8 + mt)·2 + e)·32 + l, head 4nt + (l & 3), coordinate
  //         16(l >> 2) + 2mt + e; then m[8], l[8].
  {
    float* cw = reinterpret_cast<float*>(my_stage);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float l = l_run[nt];
      l += __shfl_xor_sync(kFull, l, 4);
      l += __shfl_xor_sync(kFull, l, 8);
      l += __shfl_xor_sync(kFull, l, 16);
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        cw[((nt * 8 + mt) * 2 + 0) * 32 + lane] = o[mt][nt][0] + o[mt][nt][1];
        cw[((nt * 8 + mt) * 2 + 1) * 32 + lane] = o[mt][nt][2] + o[mt][nt][3];
      }
      if (g == 0 && 4 * nt + t < G) {
        cw[NT * 512 + 4 * nt + t] = m_run[nt];
        cw[NT * 512 + 8 + 4 * nt + t] = l;
      }
    }
  }
  __syncthreads();
  // 4a. factors f_w = 2^(m_w - M) of the warps, M and Σ_w f_w·l_w per head
  float* fw = qhat;  // [W][G]; the rotated queries are in the fragments now
  if (tid < W * G) {
    const int w = tid / G, h = tid % G;
    float M = -INFINITY;
#pragma unroll
    for (int w2 = 0; w2 < W; ++w2) M = fmaxf(M, reinterpret_cast<const float*>(stage + w2 * L.wreg)[NT * 512 + h]);
    const float mv = reinterpret_cast<const float*>(stage + w * L.wreg)[NT * 512 + h];
    fw[tid] = (mv == -INFINITY) ? 0.f : ex2(mv - M);
    if (w == 0) cM[h] = M;
  }
  __syncthreads();
  if (tid < G) {
    float Lw = 0.f;
#pragma unroll
    for (int w = 0; w < W; ++w)
      Lw = fmaf(fw[w * G + tid], reinterpret_cast<const float*>(stage + w * L.wreg)[NT * 512 + 8 + tid], Lw);
    cL[tid] = Lw;
  }
  for (int e = tid; e < NT * 512; e += NTH) {
    const int h = 4 * (e >> 9) + (e & 3);
    if (h < G) {
      float A = 0.f;
#pragma unroll
      for (int w = 0; w < W; ++w) A = fmaf(fw[w * G + h], reinterpret_cast<const float*>(stage + w * L.wreg)[e], A);
      cpart[e] = A;
    }
  }
  __syncthreads();
  // 4b. Πᵀ·acc: warp w sums its RPW rows k of Π_V, lane its 4 output coordinates
  {  // partial outputs [G][128] of warp w at the start of its region (its state is merged)
    cp_async_wait_all();
    __syncwarp();
    const float4* prow = reinterpret_cast<const float4*>(my_stage + pi_off(G));
    float4 op[G];
#pragma unroll
    for (int h = 0; h < G; ++h) op[h] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
      const int k = warp * RPW + r;  // coordinate 16gk + 2mtk + ek
      const int base = (((k >> 1) & 7) * 2 + (k & 1)) * 32 + 4 * (k >> 4);
      const float4 pv4 = prow[r * 32 + lane];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float a = cpart[(h >> 2) * 512 + base + (h & 3)];
        op[h].x = fmaf(pv4.x, a, op[h].x);
        op[h].y = fmaf(pv4.y, a, op[h].y);
        op[h].z = fmaf(pv4.z, a, op[h].z);
        op[h].w = fmaf(pv4.w, a, op[h].w);
      }
    }
#pragma unroll
    for (int h = 0; h < G; ++h) reinterpret_cast<float4*>(my_stage + h * 512)[lane] = op[h];
  }
  __syncthreads();
  for (int e = tid; e < G * 128; e += NTH) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < W; ++w) s += reinterpret_cast<const float*>(stage + w * L.wreg)[e];
    outp[e] = s;
  }
  __syncthreads();
  float* outg = p.out + ((int64_t)b * p.Hq + kvh * G) * 128;  // [G][128] of this KV head
  if (p.S == 1) {
    for (int e = tid; e < G * 128; e += NTH) outg[e] = outp[e] / cL[e >> 7];
    return;
  }
  // ---- 5. publish (m, l, Πᵀ·acc); the last CTA of the (batch, KV head) merges
  {
    float* dst = p.part + ((size_t)grp * p.S + split) * G * kPart;
    for (int e = tid; e < G * kPart; e += NTH) {
      const int h = e / kPart, k = e % kPart;
      dst[e] = k == 0 ? cM[h] : (k == 1 ? cL[h] : (k < 4 ? 0.f : outp[h * 128 + k - 4]));
    }
    __syncthreads();
    if (tid == 0) {
      // releases the CTA's stores above (ordered by the barrier); the last
      // arrival acquires everyone else's
      const int old = atomic_add_acq_rel(p.counters + grp, 1);
      const int last = old == p.S - 1;
      if (last) p.counters[grp] = 0;  // ready for the next call
      *flag = last;
    }
    __syncthreads();
  }
  if (!*flag) return;
  // all S partials into shared memory in one round trip (the tables and the ring are dead)
  float* mb = reinterpret_cast<float*>(smem);  // [S][G][kPart]
  {
    const float4* src4 = reinterpret_cast<const float4*>(p.part + (size_t)grp * p.S * G * kPart);
    const int n4 = p.S * G * (kPart / 4);
    for (int e0 = tid; e0 < n4; e0 += 8 * NTH) {
      float4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (e0 + u * NTH < n4) v[u] = __ldcg(src4 + e0 + u * NTH);
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (e0 + u * NTH < n4) reinterpret_cast<float4*>(mb)[e0 + u * NTH] = v[u];
    }
  }
  __syncthreads();
  // factor 2^(m_s - M) of every partial, into its first pad slot
  for (int e = tid; e < p.S * G; e += NTH) {
    const int h = e % G;
    float M = -INFINITY;
    for (int sp = 0; sp < p.S; ++sp) M = fmaxf(M, mb[(sp * G + h) * kPart]);
    const float ms = mb[e * kPart];
    mb[e * kPart + 2] = (ms == -INFINITY) ? 0.f : ex2(ms - M);
  }
  __syncthreads();
  for (int e = tid; e < G * 128; e += NTH) {
    const int h = e >> 7, dim = e & 127;
    float A = 0.f, Ls = 0.f;
    for (int sp = 0; sp < p.S; ++sp) {
      const float* ps = mb + (sp * G + h) * kPart;
      A = fmaf(ps[2], ps[4 + dim], A);
      Ls = fmaf(ps[2], ps[1], Ls);
    }
    outg[e] = A / Ls;
  }
}

// ------------------------------------------------------------------ launch
// CTAs per (batch, KV head): the whole grid resident at once (one CTA per SM),
// and no more partials than the last CTA can stage; among those, the fewest
// CTAs that reach the smallest number of tiles per warp (a split costs about
// one tile time for the merge through memory).
static int choose_splits(int tiles, int groups, int W, bool append, int merge_cap) {
  const int smax = std::max(1, std::min(std::min(num_sms() / std::max(1, groups), tiles), merge_cap));
  int bestS = 1;
  long best = -1;
  for (int S = 1; S <= smax; ++S) {
    // largest share of a CTA: ceil of the mean share (the owner's is smaller)
    const int worst = (!append || S == 1) ? (tiles + S - 1) / S : (2 * tiles + 2 * S - 2) / (2 * S - 1);
    const long cost = (worst + W - 1) / W + (S > 1 ? 1 : 0);
    if (best < 0 || cost < best) {
      best = cost;
      bestS = S;
    }
  }
  return bestS;
}

template <int BK, int BV, int G, bool Q = false, bool MX = false>
static cudaError_t run_step(const StepParams& p, int groups, cudaStream_t st) {
  constexpr int W = G >= 8 ? 8 : 16;
  // the short-loop variant for plain MSE caches with up to 4 query heads per KV head
  constexpr bool kHasShort = !Q && !MX && G <= 4;
  auto kern = decode_step_kernel<BK, BV, G, W, Q, MX>;
  auto kern_short = decode_step_kernel<BK, BV, G, W, Q, MX, kHasShort>;
  static PerDeviceValue smem_attr, smem_attr_short;  // set once per device, before any stream capture
  cudaError_t e = smem_attr_once(smem_attr, (const void*)kern, 227 * 1024);
  if (e == cudaSuccess && kHasShort) e = smem_attr_once(smem_attr_short, (const void*)kern_short, 227 * 1024);
  if (e != cudaSuccess) return e;
  const StepSmem L = step_smem(BK, BV, G, W, p.same_lut != 0, Q, MX);
  StepParams pp = p;
  pp.S = choose_splits(p.tiles, groups, W, p.append != 0, L.mw / (G * kPart * 4));
  // largest share of a CTA in tiles (the owner's is smaller), per warp
  const int per_warp = ((p.tiles + pp.S - 1) / pp.S + W - 1) / W;
  if (kHasShort && per_warp <= 8) kern = kern_short;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(groups * pp.S);
  cfg.blockDim = dim3(W * 32);
  cfg.dynamicSmemBytes = L.bytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, pp);
}

template <int BK, int BV>
static cudaError_t run_step_g(const StepParams& p, int G, int groups, cudaStream_t st) {
  switch (G) {
    case 1: return run_step<BK, BV, 1>(p, groups, st);
    case 2: return run_step<BK, BV, 2>(p, groups, st);
    case 4: return run_step<BK, BV, 4>(p, groups, st);
    case 8: return run_step<BK, BV, 8>(p, groups, st);
  }
  return cudaErrorInvalidValue;
}

template <int BK>
static cudaError_t run_step_v(const StepParams& p, int bv, int G, int groups, cudaStream_t st) {
  switch (bv) {
    case 1: return run_step_g<BK, 1>(p, G, groups, st);
    case 2: return run_step_g<BK, 2>(p, G, groups, st);
    case 3: return run_step_g<BK, 3>(p, G, groups, st);
    case 4: return run_step_g<BK, 4>(p, G, groups, st);
  }
  return cudaErrorInvalidValue;
}

// Launchers of the instantiated kernels, one translation unit per group of
// key bit widths (they compile in parallel).
cudaError_t decode_run_k1(const StepParams& p, int bv, int G, int groups, cudaStream_t st);
cudaError_t decode_run_k2(const StepParams& p, int bv, int G, int groups, cudaStream_t st);
cudaError_t decode_run_k3(const StepParams& p, int bv, int G, int groups, cudaStream_t st);
cudaError_t decode_run_k4(const StepParams& p, int bv, int G, int groups, cudaStream_t st);
// Prod keys ((b−1)-bit codes bk in 1..3), G in {1, 2, 4}
cudaError_t decode_run_prod(const StepParams& p, int bk, int bv, int G, int groups, cudaStream_t st);
// K and V at b + 1/2 bits per coordinate (b in 1..3), G in {1, 2, 4, 8}
cudaError_t decode_run_mixed(const StepParams& p, int b, int G, int groups, cudaStream_t st);

}  // namespace tq
