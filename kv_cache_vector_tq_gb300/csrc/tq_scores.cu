// Inner-product scores over TurboQuant codes (d = 128), on the fifth-generation
// tensor cores.
//
// "sub-byte-kv-cache-quantization-turboquant", section 工程实现的关键路径: the
// query is rotated once (q̂ = Π·q) so that each key costs a table lookup and a
// dot product:
//   MSE : score = s · ⟨q̂, ŷ⟩ = s · Σ_i q̂_i c[idx_i] / √d
//   Prod: + s · γ · √(π/2)/d · Σ_j (S q)_j (2·bit_j − 1)        ("TurboQuant 详解",
//         section TurboQuant_prod; "turboquant-first-principles-walkthrough",
//         section 内积偏差问题与 QJL 修正器).
//
// Both sums are contractions over the same 128-wide K: the A row of a key is
// [α·c[idx_i] for its 128 coordinates | ±1 for its 128 sign bits] in fp16 (one
// operand of K = 256), the B row of a query [q̂_i/α | (S q)_j] in fp16; the two
// halves of K accumulate into separate tensor-memory columns, D_mse and D_qjl,
// so that γ is applied exactly in the epilogue:
//   score = s/√d · (D_mse + γ·√(π/2)/√d · D_qjl).
//
// Two launches per 64 queries.
//  1. scores_qprep_kernel: q̂/α and S·q per query (warp-wide row dot products),
//     written as the B operand in the tensor cores' K-major core-matrix order.
//  2. scores_kernel: a persistent CTA per SM walks tiles of 128 keys:
//       warps 0-3  decode: thread = key; codes and sign words straight from
//                  global memory (one tile ahead in registers), pair-table
//                  lookups (two codes per lookup), A rows written into one of
//                  two shared-memory stages
//       warp 4     issues 16 (MSE: 8) tcgen05.mma of M = 128 keys, N = the
//                  queries (up to 64), K = 16 into one of four accumulator
//                  pairs (D_mse, D_qjl: 2 x 64 columns) in tensor memory
//       warps 5-12 epilogue, two groups of four on alternating tiles: thread =
//                  key; reads all 64 results, returns the accumulator pair,
//                  then s/√d·(D_mse + γ'·D_qjl) as one coalesced 128-byte
//                  streaming store per query per warp (measured faster than
//                  16-byte stores after a quad transpose, and than rows staged
//                  in shared memory for the bulk-copy engine); one group's
//                  stores overlap the other's tensor-memory reads.
// 13 warps: the register file is split over the four SM sub-partitions, so a
// block of more than 16 warps could not have 128 registers per thread.
//
// Up to kSmallM queries over a few thousand MSE or Prod keys take one launch
// instead: scores_small_kernel, where each CTA rotates the queries itself and
// four threads share a key (fp32 centroids and products; at that size the two
// launches and the padding of the queries to 64 cost more than the work).
#include <algorithm>

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {

namespace {

constexpr int kQTile = 64;       // queries per scan launch (MMA N)
constexpr int kKeyTile = 128;    // keys per tile (MMA M, TMEM lanes)
constexpr int kK = 256;          // contraction: 128 coordinates + 128 sign bits
constexpr int kAStage = kKeyTile * kK * 2;  // 64 KB
constexpr int kBBytes = kQTile * kK * 2;    // 32 KB
constexpr int kSbo = (kK / 8) * 128;        // bytes between 8-row groups of an operand
constexpr int kAccBufs = 4;                 // accumulator pairs (D_mse, D_qjl) in tensor memory
constexpr int kAccCols = 2 * kQTile;        // columns per pair
constexpr int kThreads = 13 * 32;

// Byte offset of element (row r, K index k) in a K-major core-matrix operand
// with kK columns: 8x8 core matrices of 128 bytes, 128 bytes apart along K,
// kSbo bytes apart along the rows.
__host__ __device__ constexpr int core_off(int r, int k) {
  return (r >> 3) * kSbo + (k >> 3) * 128 + (r & 7) * 16 + (k & 7) * 2;
}

__device__ __forceinline__ float warp_dot4(float4 a, float4 b) {
  float x = a.x * b.x + a.y * b.y + a.z * b.z + a.w * b.w;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(kFull, x, o);
  return x;
}

// Query preparation, one block (8 warps, rows 16w..16w+15) per query: the B
// row [q̂/α | S·q] of query m in tile m/64, fp16, core-matrix order (zeros for
// the rows m >= M that pad the last tile).
__global__ void __launch_bounds__(256) scores_qprep_kernel(const DevCtx c, const float* __restrict__ q, int M,
                                                           unsigned char* __restrict__ btiles) {
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
  unsigned char* tile = btiles + (size_t)(m / kQTile) * kBBytes;
  const int row = m % kQTile;
  if (tid < kK / 2) {  // thread: K index pair 2·tid, 2·tid + 1
    const int k = 2 * tid;
    const float x0 = k < 128 ? qr[k] : (prod ? sq[k - 128] : 0.f);
    const float x1 = k < 128 ? qr[k + 1] : (prod ? sq[k - 127] : 0.f);
    *reinterpret_cast<uint32_t*>(tile + core_off(row, k)) = pack_f16x2(x0, x1);
  }
}

struct ScoreParams {
  const uint32_t* codes;
  const float* norm;
  const uint32_t* qjl;
  const float* rnorm;
  const uint32_t* lut;  // pair table: 2^(2b) fp16x2 entries α·c_k
  const uint32_t* lut_hi;  // b + 1/2 bits: the (b+1)-bit codebook's pair table (same α)
  int64_t first, N;
  int W, QW;
  const unsigned char* btile;  // this launch's B operand (kBBytes)
  int m0, mq;                  // first query, queries in this launch (<= 64)
  float inv_sd;                // 1/√d
  float gscale;                // √(π/2)/√d: γ' = γ·gscale
  float* scores;
  int* status;
  uint32_t wait_limit;
};

template <int BM, bool PROD, bool MIX>
__global__ void __launch_bounds__(kThreads, 1) scores_kernel(const ScoreParams p) {
  constexpr int E = 1 << (2 * BM);
  constexpr int EH = MIX ? 4 * E : 0;  // b + 1/2 bits: entries of the (b+1)-bit pair table
  constexpr int KS = PROD ? kK / 16 : 128 / 16;  // MMAs per tile
  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char* sA = smem;                        // 2 stages
  unsigned char* sB = smem + 2 * kAStage;
  uint32_t* lut = reinterpret_cast<uint32_t*>(sB + kBBytes);  // [E][32] replicated per lane
  uint32_t* lut_hi = lut + E * 32;                             // [EH][32] (b + 1/2 bits)
  uint64_t* bars = reinterpret_cast<uint64_t*>(lut_hi + EH * 32);
  uint64_t* a_full = bars;              // [2] 4 decode warps
  uint64_t* a_empty = bars + 2;         // [2] MMA commit
  uint64_t* acc_full = bars + 4;        // [4] MMA commit
  uint64_t* acc_empty = bars + 8;       // [4] the 4 warps of one epilogue group
  uint64_t* b_full = bars + 12;         // the B operand's bulk copy
  uint64_t* drain = bars + 13;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 14);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t ntiles = (p.N + kKeyTile - 1) / kKeyTile;

  if (tid == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&a_full[s], 4);
      mbar_init(&a_empty[s], 1);
    }
    for (int b = 0; b < kAccBufs; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);
    }
    mbar_init(b_full, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  for (int i = tid; i < E * 32; i += kThreads) lut[i] = __ldg(p.lut + (i >> 5));
  for (int i = tid; i < EH * 32; i += kThreads) lut_hi[i] = __ldg(p.lut_hi + (i >> 5));
  if (warp == 0) tmem_alloc(tmem_slot, kAccBufs * kAccCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (tid == 0) {
    mbar_arrive_expect_tx(b_full, kBBytes);
    bulk_g2s(sB, p.btile, kBBytes, b_full);
  }

  if (warp < 4) {
    // ---------------- decode: key r = 32·warp + lane of the tile, all 128 coordinates
    const int r = 32 * warp + lane;
    const uint32_t* mylut = lut + lane;
    const uint32_t* mylut_hi = lut_hi + lane;
    constexpr int CW = MIX ? 2 * (2 * BM + 1) : 4 * BM;  // code words of a key
    uint32_t cw[CW], sw[4];
    auto fetch = [&](int64_t tile) {
      const int64_t key = tile * kKeyTile + r;
      const bool ok = key < p.N;
      const int64_t v = p.first + key;
#pragma unroll
      for (int w = 0; w < CW; ++w) cw[w] = ok ? __ldg(p.codes + v * p.W + w) : 0u;
      if constexpr (PROD) {
#pragma unroll
        for (int w = 0; w < 4; ++w) sw[w] = ok ? __ldg(p.qjl + v * p.QW + w) : 0u;
      }
    };
    uint32_t i = 0;
    int64_t t = blockIdx.x;
    if (t < ntiles) fetch(t);
    for (; t < ntiles; t += gridDim.x, ++i) {
      uint32_t c[CW], sb[4];
#pragma unroll
      for (int w = 0; w < CW; ++w) c[w] = cw[w];
#pragma unroll
      for (int w = 0; w < 4; ++w) sb[w] = sw[w];
      if (t + gridDim.x < ntiles) fetch(t + gridDim.x);  // next tile's words in flight
      const uint32_t s = i & 1u;
      if (!__all_sync(kFull, bar_wait(&a_empty[s], ((i >> 1) & 1u) ^ 1u, abort_flag, p.status, p.wait_limit))) break;
      unsigned char* A = sA + s * kAStage;
      // 128 coordinates = 16 core rows of 8 fp16 (pairs from the table)
#pragma unroll
      for (int k8 = 0; k8 < 16; ++k8) {
        uint32_t v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if constexpr (MIX) {  // coordinates 8·k8.. take BM + 1 bits for even k8, BM for odd
            const int pos = mixed_pos(8 * k8 + 2 * e, BM);
            v[e] = (k8 & 1) ? mylut[get_bits<2 * BM>(c, pos) << 5] : mylut_hi[get_bits<2 * BM + 2>(c, pos) << 5];
          } else {
            v[e] = mylut[get_bits<2 * BM>(c, (8 * k8 + 2 * e) * BM) << 5];
          }
        }
        *reinterpret_cast<uint4*>(A + core_off(r, 8 * k8)) = make_uint4(v[0], v[1], v[2], v[3]);
      }
      if constexpr (PROD) {  // ±1 for 128 sign bits
#pragma unroll
        for (int k8 = 0; k8 < 16; ++k8) {
          const uint32_t byte = (sb[k8 >> 2] >> (8 * (k8 & 3))) & 0xFFu;
          // bit i of the byte at i and at i + 15: shifted left by 15 - 2e, bit
          // 2e lands on 15 and bit 2e + 1 on 31, the sign bits of the word's
          // two fp16 halves
          const uint32_t sp = byte | (byte << 15);
          uint32_t v[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)  // −1 in both halves; bit 1 flips its half to +1
            v[e] = ((sp << (15 - 2 * e)) & 0x80008000u) ^ 0xBC00BC00u;
          *reinterpret_cast<uint4*>(A + core_off(r, 128 + 8 * k8)) = make_uint4(v[0], v[1], v[2], v[3]);
        }
      }
      fence_proxy_async();  // generic-proxy stores, read next by the tensor cores
      __syncwarp();
      if (lane == 0) mbar_arrive(&a_full[s]);
    }
  } else if (warp == 4) {
    // ---------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = umma_idesc_f16(kKeyTile, kQTile);
      bool ok = bar_wait(b_full, 0u, abort_flag, p.status, p.wait_limit);
      const uint32_t bbase = smem_u32(sB);
      uint32_t i = 0;
      for (int64_t t = blockIdx.x; ok && t < ntiles; t += gridDim.x, ++i) {
        const uint32_t s = i & 1u, b = i % kAccBufs;
        if (!bar_wait(&acc_empty[b], ((i / kAccBufs) & 1u) ^ 1u, abort_flag, p.status, p.wait_limit) ||
            !bar_wait(&a_full[s], (i >> 1) & 1u, abort_flag, p.status, p.wait_limit)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t abase = smem_u32(sA + s * kAStage);
#pragma unroll
        for (int ks = 0; ks < KS; ++ks)  // K steps 0-7 into D_mse, 8-15 into D_qjl
          umma_f16(tmem + b * kAccCols + (ks >= 8 ? kQTile : 0), umma_desc(abase + ks * 256, 128, kSbo),
                   umma_desc(bbase + ks * 256, 128, kSbo), idesc, (ks & 7) > 0 ? 1u : 0u);
        umma_commit(&a_empty[s]);
        umma_commit(&acc_full[b]);
      }
      umma_commit(drain);  // every MMA issued completes before tensor memory is released
      for (uint32_t n = 0; n < kSpinLimitDev && !mbar_try_wait(drain, 0u); ++n) {
      }
    }
  } else {
    // ---------------- epilogue: group grp takes tiles i ≡ grp (mod 2); thread = key
    //                  (TMEM lane 32·(warp % 4) + lane)
    const int grp = (warp - 5) >> 2, q4 = warp & 3, r = 32 * q4 + lane;
    const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
    uint32_t i = grp;
    for (int64_t t = blockIdx.x + (int64_t)grp * gridDim.x; t < ntiles; t += 2 * (int64_t)gridDim.x, i += 2) {
      const uint32_t b = i % kAccBufs;
      const int64_t key = t * kKeyTile + r;
      const bool ok = key < p.N;
      const float sc = ok ? __ldg(p.norm + p.first + key) * p.inv_sd : 0.f;
      const float gq = (PROD && ok) ? __ldg(p.rnorm + p.first + key) * p.gscale : 0.f;
      if (!__all_sync(kFull, bar_wait(&acc_full[b], (i / kAccBufs) & 1u, abort_flag, p.status, p.wait_limit))) break;
      tc_fence_after();
      const uint32_t acc = tmem + lane_base + b * kAccCols;
      float* out = p.scores + (int64_t)p.m0 * p.N + key;
      float o0[32];  // queries 0-31, stored once the pair is returned
      uint32_t dm[32], dq[32];
      tmem_ld32_nw(acc, dm);
      if constexpr (PROD) tmem_ld32_nw(acc + kQTile, dq);
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 32; ++j)
        o0[j] = sc * (PROD ? fmaf(gq, __uint_as_float(dq[j]), __uint_as_float(dm[j])) : __uint_as_float(dm[j]));
      tmem_ld32_nw(acc + 32, dm);  // queries 32-63
      if constexpr (PROD) tmem_ld32_nw(acc + kQTile + 32, dq);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[b]);
      if (ok) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (32 + j < p.mq)
            __stcs(out + (int64_t)(32 + j) * p.N,
                   sc * (PROD ? fmaf(gq, __uint_as_float(dq[j]), __uint_as_float(dm[j])) : __uint_as_float(dm[j])));
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (j < p.mq) __stcs(out + (int64_t)j * p.N, o0[j]);
      }
    }
  }

  // the B operand's bulk copy lands before the CTA may exit, also when a wait
  // gave up before the MMA issuer saw it complete (bounded)
  if (tid == 0)
    for (uint32_t n = 0; n < kSpinLimitDev && !mbar_try_wait(b_full, 0u); ++n) {
    }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kAccBufs * kAccCols);
  }
}

constexpr int kSmallM = 8;         // queries served by scores_small_kernel
constexpr int kSmallThreads = 256;  // 64 keys per trip, four threads per key

struct SmallScoreParams {
  const float* q;  // [M][128]
  int M;
  const float* pi;     // Π, fp32 row-major
  const float* s_mat;  // Prod: S, fp32 row-major
  const uint32_t* codes;
  const float* norm;
  const uint32_t* qjl;
  const float* rnorm;
  int64_t first, N;
  int W, QW;
  float cen[16];  // centroids, unit-variance units
  float inv_sd, gscale;
  float* scores;  // [M][N]
};

// Row r (< 128) of A·q_m for every query, thread (r, half h) summing columns
// [64h, 64h + 64): partial sums into part[h][m][r].
__device__ __forceinline__ void rotate_half(const float* __restrict__ A, const float (*qs)[128], int M, int r, int h,
                                            float (*part)[kSmallM][128]) {
  float acc[kSmallM];
#pragma unroll
  for (int m = 0; m < kSmallM; ++m) acc[m] = 0.f;
  const float4* row = reinterpret_cast<const float4*>(A + (size_t)r * 128 + 64 * h);
#pragma unroll 4
  for (int i4 = 0; i4 < 16; ++i4) {
    const float4 w = __ldg(row + i4);
#pragma unroll
    for (int m = 0; m < kSmallM; ++m)
      if (m < M) {
        const float4 x = *reinterpret_cast<const float4*>(&qs[m][64 * h + 4 * i4]);
        acc[m] = fmaf(w.x, x.x, fmaf(w.y, x.y, fmaf(w.z, x.z, fmaf(w.w, x.w, acc[m]))));
      }
  }
#pragma unroll
  for (int m = 0; m < kSmallM; ++m)
    if (m < M) part[h][m][r] = acc[m];
}

// Scores of M <= kSmallM queries in one launch.  Every CTA first rotates the
// queries (q̂ = Π·q and, for Prod, S·q; thread (row, column half)), then walks
// the keys 64 at a time: thread group g of four takes key g, thread j of the
// group its 32 coordinates [32j, 32j + 32), i.e. BM whole words of the key's
// stream (and, for Prod, its sign word j); Σ c[idx]·q̂ (and Σ ±(S·q)) over
// them, two shuffles across the group, s/√d·(D_mse + γ·√(π/2)/√d·D_qjl).
template <int BM, bool PROD>
__global__ void __launch_bounds__(kSmallThreads, 2) scores_small_kernel(const SmallScoreParams p) {
  __shared__ __align__(16) float qs[kSmallM][128];
  __shared__ __align__(16) float part[2][kSmallM][128];
  __shared__ float qh[kSmallM][4][33];  // q̂ by coordinate group, padded: the four groups on distinct banks
  __shared__ float sqh[PROD ? kSmallM : 1][4][33];
  __shared__ float cen[16];
  const int tid = threadIdx.x, M = p.M;
  for (int e = tid; e < M * 128; e += kSmallThreads) qs[e >> 7][e & 127] = __ldg(p.q + e);
  if (tid < 16) cen[tid] = p.cen[tid];
  __syncthreads();
  const int r = tid & 127, h = tid >> 7;
  rotate_half(p.pi, qs, M, r, h, part);
  __syncthreads();
#pragma unroll
  for (int m = 0; m < kSmallM; ++m)
    if (m < M && h == 0) qh[m][r >> 5][r & 31] = part[0][m][r] + part[1][m][r];
  if constexpr (PROD) {
    __syncthreads();
    rotate_half(p.s_mat, qs, M, r, h, part);
    __syncthreads();
#pragma unroll
    for (int m = 0; m < kSmallM; ++m)
      if (m < M && h == 0) sqh[m][r >> 5][r & 31] = part[0][m][r] + part[1][m][r];
  }
  __syncthreads();
  const int j = tid & 3;
  for (int64_t base = (int64_t)blockIdx.x * (kSmallThreads / 4); base < p.N;
       base += (int64_t)gridDim.x * (kSmallThreads / 4)) {
    const int64_t key = base + (tid >> 2);
    const bool ok = key < p.N;
    const int64_t v = p.first + (ok ? key : 0);
    uint32_t w[BM];
#pragma unroll
    for (int k = 0; k < BM; ++k) w[k] = ok ? __ldg(p.codes + v * p.W + j * BM + k) : 0u;
    float acc[kSmallM], accq[kSmallM];
#pragma unroll
    for (int m = 0; m < kSmallM; ++m) acc[m] = accq[m] = 0.f;
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      const float cv = cen[get_bits<BM>(w, c * BM)];
#pragma unroll
      for (int m = 0; m < kSmallM; ++m)
        if (m < M) acc[m] = fmaf(cv, qh[m][j][c], acc[m]);
    }
    float sc = 0.f, gq = 0.f;
    if (ok) {
      sc = __ldg(p.norm + v) * p.inv_sd;
      if constexpr (PROD) gq = __ldg(p.rnorm + v) * p.gscale;
    }
    if constexpr (PROD) {
      const uint32_t sg = ok ? __ldg(p.qjl + v * p.QW + j) : 0u;
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const uint32_t neg = ((sg >> c) & 1u) ? 0u : 0x80000000u;  // bit 0: −(S·q)_c
#pragma unroll
        for (int m = 0; m < kSmallM; ++m)
          if (m < M) accq[m] += __uint_as_float(__float_as_uint(sqh[m][j][c]) ^ neg);
      }
    }
#pragma unroll
    for (int m = 0; m < kSmallM; ++m) {
      if (m >= M) break;
      float a = PROD ? fmaf(gq, accq[m], acc[m]) : acc[m];
      a += __shfl_xor_sync(kFull, a, 1);
      a += __shfl_xor_sync(kFull, a, 2);
      if (ok && j == 0) p.scores[(int64_t)m * p.N + key] = sc * a;
    }
  }
}

template <int BM, bool PROD>
cudaError_t run_scores_small(const SmallScoreParams& p, cudaStream_t st) {
  const int64_t trips = (p.N + kSmallThreads / 4 - 1) / (kSmallThreads / 4);
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(trips, 2 * (int64_t)num_sms()));
  scores_small_kernel<BM, PROD><<<grid, kSmallThreads, 0, st>>>(p);
  return cudaGetLastError();
}

template <int BM, bool PROD, bool MIX = false>
cudaError_t run_scores(const ScoreParams& p, cudaStream_t st) {
  constexpr int E = 1 << (2 * BM);
  constexpr size_t smem = 2 * kAStage + kBBytes + (MIX ? 5 : 1) * E * 32 * 4 + 256;
  auto k = scores_kernel<BM, PROD, MIX>;
  static PerDeviceValue attr;  // set once per device, outside any later stream capture
  const cudaError_t e = smem_attr_once(attr, (const void*)k, (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t tiles = (p.N + kKeyTile - 1) / kKeyTile;
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(tiles, (int64_t)num_sms()));
  k<<<grid, kThreads, smem, st>>>(p);
  return cudaGetLastError();
}

}  // namespace

size_t scores_ws_bytes(const DevCtx& c, int M) {
  (void)c;
  return (size_t)((M + kQTile - 1) / kQTile) * kBBytes + 256;
}

tq_status launch_scores(const DevCtx& c, const float* q, int M, const tq_codes* keys, int64_t first,
                        int64_t N, float* scores, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (c.d != 128) return TQ_ERR_UNSUPPORTED;
  if (ws_bytes < scores_ws_bytes(c, M)) return TQ_ERR_INVALID_ARG;
  // the one-launch scorer while its per-key cost (which grows with M) stays
  // below the fixed cost of the tensor-core path (measured: one query, 4096
  // keys 11.7 against 16.6 us, 65536 keys 21.8 against 19.9 us)
  if (M <= kSmallM && N * (M + 2) <= 98304 && (c.mode == TQ_MSE || c.mode == TQ_PROD)) {
    SmallScoreParams sp;
    sp.q = q;
    sp.M = M;
    sp.pi = c.pi;
    sp.s_mat = c.s_mat;
    sp.codes = keys->d_codes;
    sp.norm = keys->d_norm;
    sp.qjl = keys->d_qjl;
    sp.rnorm = keys->d_rnorm;
    sp.first = first;
    sp.N = N;
    sp.W = c.words_per_vec;
    sp.QW = c.qjl_words_per_vec;
    for (int k = 0; k < 16; ++k) sp.cen[k] = c.cen[k];
    sp.inv_sd = 1.f / c.sqrt_d;
    sp.gscale = (float)(1.2533141373155002 / std::sqrt((double)c.d));
    sp.scores = scores;
    const bool prod = c.mode == TQ_PROD;
    cudaError_t e = cudaErrorInvalidValue;
    switch (c.b_mse) {
      case 1: e = prod ? run_scores_small<1, true>(sp, stream) : run_scores_small<1, false>(sp, stream); break;
      case 2: e = prod ? run_scores_small<2, true>(sp, stream) : run_scores_small<2, false>(sp, stream); break;
      case 3: e = prod ? run_scores_small<3, true>(sp, stream) : run_scores_small<3, false>(sp, stream); break;
      case 4: e = run_scores_small<4, false>(sp, stream); break;
      default: return TQ_ERR_UNSUPPORTED;
    }
    return e == cudaSuccess ? TQ_OK : set_cuda_error(e);
  }
  unsigned char* bt = static_cast<unsigned char*>(ws);
  const int nqt = (M + kQTile - 1) / kQTile;
  scores_qprep_kernel<<<nqt * kQTile, 256, 0, stream>>>(c, q, M, bt);  // rows past M written as zeros
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_cuda_error(e);
  ScoreParams p;
  p.codes = keys->d_codes;
  p.norm = keys->d_norm;
  p.qjl = keys->d_qjl;
  p.rnorm = keys->d_rnorm;
  p.lut = c.lut;
  p.lut_hi = c.lut_hi;
  p.first = first;
  p.N = N;
  p.W = c.words_per_vec;
  p.QW = c.qjl_words_per_vec;
  p.inv_sd = 1.f / c.sqrt_d;
  p.gscale = (float)(1.2533141373155002 / std::sqrt((double)c.d));
  p.scores = scores;
  p.status = c.status;
  p.wait_limit = c.wait_limit;
  const bool prod = c.mode == TQ_PROD;
  for (int m0 = 0; m0 < M; m0 += kQTile) {
    p.m0 = m0;
    p.mq = std::min(kQTile, M - m0);
    p.btile = bt + (size_t)(m0 / kQTile) * kBBytes;
    if (c.mode == TQ_MIXED) {
      switch (c.b_mse) {
        case 1: e = run_scores<1, false, true>(p, stream); break;
        case 2: e = run_scores<2, false, true>(p, stream); break;
        case 3: e = run_scores<3, false, true>(p, stream); break;
        default: return TQ_ERR_UNSUPPORTED;
      }
      if (e != cudaSuccess) return set_cuda_error(e);
      continue;
    }
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
