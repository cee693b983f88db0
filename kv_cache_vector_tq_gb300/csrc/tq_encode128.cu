// TurboQuant encoder for d = 128 (MSE and Prod, fp32 or fp16 rows, TOKEN or
// PAIR layout) on the fifth-generation tensor cores.
//
// "TurboQuant 详解", section 一个具体例子：KV Cache 在 prefill 和 decode 里怎么量化
// steps 1-6 (s = ‖x‖, y = Π·x/s, idx_i = nearest centroid of √d·y_i, pack the
// indices, store s) and section TurboQuant_prod (a (b-1)-bit MSE stage, the
// residual r = u − Πᵀŷ, γ = ‖r‖ and the 1-bit code sign(S·r), sign(0) = +1);
// the rotation is the encoder's one dense matrix product ("turboquant-first-
// principles-walkthrough", section 通用码本设计).
//
// A persistent CTA per SM walks tiles of 128 rows.  Per tile the rotation is
// Y = X·(pi_scale·Π)ᵀ as tcgen05.mma of M = N = 128 and K = 16, eight K steps
// per pass, into one fp32 accumulator in tensor memory:
//   fp16 rows: A is the x tile itself, loaded by TMA in the 128-byte swizzle
//              and read by the MMA from shared memory (x is exact in fp16);
//              two passes, x·Πlo then x·Πhi.
//   fp32 rows: A is x·2^e split into fp16 hi + lo (2^e puts s·2^e in [16, 32)),
//              written to tensor memory by the prep warps; three passes,
//              xl·Πhi, xh·Πlo, then xh·Πhi.
// The low-order passes go first so that their small products are not
// truncated against a large accumulator.  The tensor cores' fp32 accumulation
// still truncates (measured on GB300 about 7e-9·L in v units over an
// accumulated K range L, ~1e-6 at L = 128), so every coordinate within 8e-6 of
// a threshold is recomputed by one warp as a float-float dot product of the
// input row with the fp32 Π (error ~3e-8) and decided again: codes match the
// fp64 definition outside the 1e-6 band, as on every other path.
// Prod: the epilogue forms r_rot = (v − c[idx])/√d per coordinate (γ = ‖r_rot‖
// = ‖r‖, Π being orthogonal), writes it scaled by 2^e (γ·2^e in [16, 32)) as
// fp16 hi + lo into tensor memory, and a second three-pass product with
// (m_scale·S·Πᵀ) gives p = S·r up to a positive factor; bit_j = [p_j >= 0].
//
// Warp roles (22 warps):
//   0     producer: the B operand tables once (bulk copy), then per tile one
//         2-D TMA load per 128-byte column box of the x tile.
//   1     MMA issuer (one thread).
//   2-5   prep: thread = row = TMEM lane (warp w owns lanes 32·(w % 4)..+31):
//         s = ‖x‖ from the staged tile (fp32 sums; a row whose sum leaves
//         (1e-30, 1e36) is summed again scaled by a power of two); fp32 rows:
//         the split A operand into tensor memory.
//   6-21  epilogue: thread = row, four warps per TMEM lane quadrant, each for
//         one 32-column chunk (its codes are BM whole words of the row's
//         stream; at b + 1/2 bits 2·BM + 1 halfwords): v = acc·√d/(s·scales),
//         bucketize (a branch-free count over the thresholds, kept as kernel
//         constants) with a near-threshold flag, pack in registers, recompute
//         flagged coordinates, store; Prod: γ over the four chunks, the
//         chunk's residual operand, the second product, its sign bits.
// All waits are bounded (tq_ctx_set_wait_limit); a wait that gives up sets the
// abort flag, which every role polls, and bit 0 of the status word.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {

namespace {

constexpr int kRows = 128;                   // rows per tile = TMEM lanes = MMA M
constexpr int kDim = 128;                    // d = MMA N = K
constexpr int kBox = kRows * 128;            // one 128-byte column box of the x tile: 16 KB
constexpr int kTab = 4 * kUmmaPlaneBytes;    // B operand of one 128 x 128 matrix: (hi, lo) x 2 K chunks
// 16 epilogue warps, one 32-column chunk of a tensor-memory lane quadrant each
// (22 warps in all)
constexpr int kEpiWarps = 16;
constexpr int kEncThreads = (6 + kEpiWarps) * 32;
constexpr float kMargin = 8e-6f;             // recomputation band around each threshold (v units)

template <bool F16, bool PROD>
struct Lay {
  static constexpr int ES = F16 ? 2 : 4;
  static constexpr int Boxes = kDim * ES / 128;  // 2 (fp16) or 4 (fp32)
  static constexpr int Stage = Boxes * kBox;     // 32 or 64 KB
  static constexpr int XStages = F16 ? (PROD ? 2 : 3) : (PROD ? 1 : 2);
  static constexpr int AStages = F16 ? 0 : (PROD ? 1 : 2);  // fp32: split A in tensor memory
  static constexpr int AccBufs = (PROD && !F16) ? 1 : 2;
  // tensor memory columns: A stages (hi 64 | lo 64), accumulators, then (Prod)
  // the residual operand (hi 64 | lo 64) and the QJL accumulator
  static constexpr uint32_t ColAcc = AStages * 128;
  static constexpr uint32_t ColA2 = ColAcc + AccBufs * 128;
  static constexpr uint32_t ColAcc2 = ColA2 + 128;
  static constexpr uint32_t Cols = PROD ? ColAcc2 + 128 : ColA2;
  static constexpr uint32_t TmemCols = Cols <= 256 ? 256 : 512;
  static constexpr int OffX = kTab * (PROD ? 2 : 1);
  static constexpr int OffNorm = OffX + XStages * Stage;
  static constexpr int OffThr = OffNorm + (AccBufs + 8) * kRows * 4;  // norms, then (Prod) γ² per chunk
  static constexpr int OffCen = OffThr + 16 * 4;
  static constexpr int OffBar = OffCen + 16 * 4;
  static constexpr int NBar = 26;
  static constexpr int Smem = OffBar + NBar * 8 + 16;
  static constexpr int SmemAlloc = Smem + 1024;  // slack to align the base to 1024 bytes
  static_assert(Cols <= 512, "tensor memory");
  static_assert(SmemAlloc <= 227 * 1024, "shared memory");
};

struct Enc128Params {
  const void* x;
  int64_t N;
  uint32_t* codes;
  float* norm;
  uint32_t* qjl;
  float* rnorm;
  const unsigned char* tab_pi;  // pi_scale·Π as B tiles (hi, lo planes per 64-wide K chunk)
  const unsigned char* tab_m;   // Prod: m_scale·S·Πᵀ in the same layout
  const float* pi;              // Π, fp32 row-major (recomputation)
  float pi_scale;
  double sqrt_d;   // recomputation (rare) in fp64
  float sqrt_df;
  float thr[15];
  float cen[16];
  float thr_hi[15];  // b + 1/2 bits: the (BM+1)-bit codebook's thresholds
  int layout, W, QW, pair_aligned;
  int64_t offset, group_rows, group_stride;
  int* status;
  uint32_t wait_limit;
};

// Destination vector of row r (< N <= 2^31 - 1): 32-bit division only.
__device__ __forceinline__ int64_t dest_row(const Enc128Params& p, int64_t r) {
  if (p.group_rows >= p.N) return p.offset + r;
  const uint32_t rr = (uint32_t)r, gr = (uint32_t)p.group_rows, gq = rr / gr;
  return (int64_t)gq * p.group_stride + p.offset + (int64_t)(rr - gq * gr);
}

// Branch-free bucketize against thresholds held as kernel constants (every
// index is known at compile time, so no shared-memory loads and no dependent
// chain): code = #{k : v >= t_k}, near = v lies within m of some threshold.
// The codebooks this kernel serves are symmetric (the ones tq_codebook_build
// makes), so |v| is compared with the H = 2^(BM-1) - 1 positive thresholds
// only; a value exactly equal to a negative threshold then counts as below
// it, which differs from the definition only at exact ties, all inside the
// band that parity excuses.
template <int BM>
__device__ __forceinline__ uint32_t bucketize_c(float v, const float (&thr)[15], float m, bool& near) {
  constexpr int H = (1 << (BM - 1)) - 1;
  const float a = fabsf(v);
  float dmin = a;
  int n = 0;
#pragma unroll
  for (int j = 0; j < H; ++j) {
    const float dj = a - thr[H + 1 + j];
    dmin = fminf(dmin, fabsf(dj));
    n += dj >= 0.f ? 1 : 0;
  }
  near = dmin < m;
  return v >= 0.f ? (uint32_t)(H + 1 + n) : (uint32_t)(H - n);
}

// Symmetric bucketize without a per-coordinate near test: code of v from the
// sign bits of |v| - t over the positive thresholds (a sign bit counts a
// threshold above |v|, one shift-add each), and every |v - t| (and |v|, for
// the threshold at 0) folded into dmin, a running minimum over the chunk.
template <int BM>
__device__ __forceinline__ uint32_t bucketize_fold(float v, const float (&thr)[15], float& dmin) {
  constexpr int H = (1 << (BM - 1)) - 1;
  constexpr uint32_t kAll = (1u << BM) - 1u;  // 2H + 1
  const float a = fabsf(v);
  dmin = fminf(dmin, a);
  uint32_t above = 0u;  // thresholds t > |v|
#pragma unroll
  for (int j = 0; j < H; ++j) {
    const float dj = a - thr[H + 1 + j];
    dmin = fminf(dmin, fabsf(dj));
    above += __float_as_uint(dj) >> 31;
  }
  // v >= 0: H + 1 + (H - above) = kAll - above; v < 0: H - (H - above) = above
  // = (kAll - above) ^ kAll
  return (kAll - above) ^ ((uint32_t)((int32_t)__float_as_uint(v) >> 31) & kAll);
}

// Positive thresholds of a symmetric BM-bit codebook (one slot at BM = 1).
template <int BM>
constexpr int kTB = BM == 1 ? 1 : (1 << (BM - 1)) - 1;

// Symmetric bucketize of an accumulator value x against the positive
// thresholds tb, already divided by the row's scale (x·scale >= t and x >= tb
// differ only by roundings far inside the recomputation band): bucketize_fold
// without the per-coordinate scaling.  (A binary search over tb, with the
// bracketing thresholds' distances, issued fewer compares but ran slower.)
template <int BM>
__device__ __forceinline__ uint32_t bucketize_sc(float x, const float (&tb)[kTB<BM>], float& dmin) {
  constexpr int H = (1 << (BM - 1)) - 1;
  constexpr uint32_t kAll = (1u << BM) - 1u;
  const float a = fabsf(x);
  dmin = fminf(dmin, a);
  uint32_t above = 0u;
#pragma unroll
  for (int j = 0; j < H; ++j) {
    const float dj = a - tb[j];
    dmin = fminf(dmin, fabsf(dj));
    above += __float_as_uint(dj) >> 31;
  }
  return (kAll - above) ^ ((uint32_t)((int32_t)__float_as_uint(x) >> 31) & kAll);
}

// The row's positive thresholds divided by its scale: tb[j] = t_{H+1+j}·inv.
template <int BM>
__device__ __forceinline__ void scaled_thresholds(const float (&thr)[15], float inv, float (&tb)[kTB<BM>]) {
  constexpr int H = (1 << (BM - 1)) - 1;
#pragma unroll
  for (int j = 0; j < kTB<BM>; ++j) tb[j] = BM == 1 ? 0.f : thr[H + 1 + j] * inv;
}

// One 32-column chunk of plain MSE codes (symmetric codebook) from the raw
// accumulator: BM code words (coordinate j at bits j·BM), and `flagged` when a
// coordinate lies within mg (the band in accumulator units) of a threshold.
template <int BM>
__device__ __forceinline__ void chunk_codes_s(const uint32_t (&a)[32], const float (&tb)[kTB<BM>], float mg,
                                              uint32_t (&cw)[BM], bool& flagged) {
#pragma unroll
  for (int w = 0; w < BM; ++w) cw[w] = 0u;
  float dmin = INFINITY;
#pragma unroll
  for (int j = 0; j < 32; ++j) put_bits<BM>(cw, j * BM, bucketize_sc<BM>(__uint_as_float(a[j]), tb, dmin));
  flagged = dmin < mg;
}

// Near-threshold flags of a chunk (symmetric codebook), bit j for coordinate j.
template <int BM>
__device__ __forceinline__ uint32_t near_mask(const uint32_t (&a)[32], float f, const float (&thr)[15]) {
  uint32_t m32 = 0u;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    bool near;
    bucketize_c<BM>(__uint_as_float(a[j]) * f, thr, kMargin, near);
    m32 |= (near ? 1u : 0u) << j;
  }
  return m32;
}

// One 32-column chunk of the Prod encoder's (b-1)-bit MSE stage: its BM code
// words (coordinate j at bits j·BM), the sum of squared residuals in v units
// (for γ), and `flagged` when a coordinate of the chunk lies near a threshold
// (the caller finds which in the rare chunks that have one).
template <int BM>
__device__ __forceinline__ void prod_chunk_codes(const uint32_t (&a)[32], float f, const float (&thr)[15],
                                                 const float* cen_s, uint32_t (&cw)[BM], float& g2,
                                                 bool& flagged) {
#pragma unroll
  for (int w = 0; w < BM; ++w) cw[w] = 0u;
  float dmin = INFINITY;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const float v = __uint_as_float(a[j]) * f;
    const uint32_t code = bucketize_fold<BM>(v, thr, dmin);
    put_bits<BM>(cw, j * BM, code);
    const float rr = v - cen_s[code];
    g2 = fmaf(rr, rr, g2);
  }
  flagged = dmin < kMargin;
}

// b + 1/2 bits per coordinate: coordinate j (0..31) of a 32-column chunk has
// BM + 1 bits where j mod 16 < 8 and BM bits elsewhere; its code starts at bit
// mixed_pos(j, BM) of the chunk's codes (every 16 coordinates span 8·(2·BM + 1)
// bits, so a chunk is 2·BM + 1 halfwords of the row's stream).
// One chunk at b + 1/2 bits (symmetric codebooks): codes into hw at
// compile-time positions; a coordinate near a threshold anywhere in the chunk
// sets `flagged`.
template <int BM>
__device__ __forceinline__ void mix_chunk_codes(const uint32_t (&a)[32], const float (&tlo)[kTB<BM>],
                                                const float (&thi)[kTB<BM + 1>], float mg, uint32_t (&hw)[BM + 1],
                                                bool& flagged) {
  float dmin = INFINITY;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const float x = __uint_as_float(a[j]);
    if ((j & 8) == 0)
      put_bits<BM + 1>(hw, mixed_pos(j, BM), bucketize_sc<BM + 1>(x, thi, dmin));
    else
      put_bits<BM>(hw, mixed_pos(j, BM), bucketize_sc<BM>(x, tlo, dmin));
  }
  flagged = dmin < mg;
}

// BM consecutive words to dst (4-byte aligned) in the widest aligned vector
// stores: one lane's codes of a chunk are contiguous, and every store
// instruction of a warp touches a sector per lane, so fewer, wider stores
// write fewer partial sectors.
template <int BM>
__device__ __forceinline__ void store_words(uint32_t* dst, const uint32_t (&w)[BM]) {
  const uint32_t al = (uint32_t)reinterpret_cast<uintptr_t>(dst) & 15u;
  if constexpr (BM == 1) {
    dst[0] = w[0];
  } else if constexpr (BM == 2) {
    if ((al & 7u) == 0u) {
      *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
    } else {
      dst[0] = w[0];
      dst[1] = w[1];
    }
  } else if constexpr (BM == 3) {
    if ((al & 7u) == 0u) {
      *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
      dst[2] = w[2];
    } else {
      dst[0] = w[0];
      *reinterpret_cast<uint2*>(dst + 1) = make_uint2(w[1], w[2]);
    }
  } else {
    if (al == 0u) {
      *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
    } else if ((al & 7u) == 0u) {
      *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
      *reinterpret_cast<uint2*>(dst + 2) = make_uint2(w[2], w[3]);
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k) dst[k] = w[k];
    }
  }
}

// 2·BM + 1 halfwords h (the low ones of words w[0..BM]) to halfword address
// dst: word stores where the start is word-aligned, else one halfword first
// (fewer partial-sector writes than one store per halfword).
template <int BM>
__device__ __forceinline__ void store_halfwords(uint16_t* dst, const uint32_t (&w)[BM + 1]) {
  uint32_t v[BM];
  if ((reinterpret_cast<uintptr_t>(dst) & 3u) == 0u) {
#pragma unroll
    for (int k = 0; k < BM; ++k) v[k] = w[k];
    store_words<BM>(reinterpret_cast<uint32_t*>(dst), v);
    dst[2 * BM] = (uint16_t)w[BM];
  } else {
    dst[0] = (uint16_t)w[0];
#pragma unroll
    for (int k = 0; k < BM; ++k) v[k] = __funnelshift_r(w[k], w[k + 1], 16);
    store_words<BM>(reinterpret_cast<uint32_t*>(dst + 1), v);
  }
}

// Half (16 coordinates) of a b + 1/2-bit chunk: codes at mixed_pos(j, BM) of
// a 64-bit group (8·(2·BM + 1) bits), distances folded into dmin.
template <int BM>
__device__ __forceinline__ uint64_t mix_half_codes(const uint32_t (&a)[16], const float (&tlo)[kTB<BM>],
                                                   const float (&thi)[kTB<BM + 1>], float& dmin) {
  uint32_t w[2] = {0u, 0u};
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const float x = __uint_as_float(a[j]);
    if ((j & 8) == 0)
      put_bits<BM + 1>(w, mixed_pos(j, BM), bucketize_sc<BM + 1>(x, thi, dmin));
    else
      put_bits<BM>(w, mixed_pos(j, BM), bucketize_sc<BM>(x, tlo, dmin));
  }
  return (uint64_t)w[0] | ((uint64_t)w[1] << 32);
}

// Near-threshold flags of a b + 1/2-bit chunk, each coordinate against its own codebook.
template <int BM>
__device__ __forceinline__ uint32_t mix_near_mask(const uint32_t (&a)[32], float f, const float (&tlo)[15],
                                                  const float (&thi)[15]) {
  uint32_t m32 = 0u;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const float v = __uint_as_float(a[j]) * f;
    bool near;
    if ((j & 8) == 0)
      bucketize_c<BM + 1>(v, thi, kMargin, near);
    else
      bucketize_c<BM>(v, tlo, kMargin, near);
    m32 |= (near ? 1u : 0u) << j;
  }
  return m32;
}

// One 32-column chunk (symmetric codebook) for the PAIR layout: coordinate j's
// code goes straight to its even-vector slot of the chunk's pair block, bits
// 2(j mod 16)·BM of lo (j < 16) or hi (j >= 16), so that a row pair's block
// words are one exchange and an OR away (an odd vector shifts by BM first).
template <int BM>
__device__ __forceinline__ void chunk_codes_pair(const uint32_t (&a)[32], const float (&tb)[kTB<BM>], float mg,
                                                 uint32_t (&lo)[BM], uint32_t (&hi)[BM], bool& flagged) {
#pragma unroll
  for (int w = 0; w < BM; ++w) lo[w] = hi[w] = 0u;
  float dmin = INFINITY;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const uint32_t code = bucketize_sc<BM>(__uint_as_float(a[j]), tb, dmin);
    if (j < 16)
      put_bits<BM>(lo, 2 * j * BM, code);
    else
      put_bits<BM>(hi, 2 * (j - 16) * BM, code);
  }
  flagged = dmin < mg;
}

// Words x << BM (BM < 32) of a BM-word array, the top field leaving nothing behind
// (slot 30 of the even vector moves to slot 31).
template <int BM>
__device__ __forceinline__ void shift_slot(uint32_t (&x)[BM]) {
#pragma unroll
  for (int w = BM - 1; w > 0; --w) x[w] = (x[w] << BM) | (x[w - 1] >> (32 - BM));
  x[0] <<= BM;
}

// Bits [pos, pos + width) of a word array (run-time position and width), and their replacement.
template <int N>
__device__ __forceinline__ uint32_t get_bits_rt(const uint32_t (&wd)[N], int pos, int width) {
  uint32_t v = 0;
#pragma unroll
  for (int w = 0; w < N; ++w) {
    const int sh = pos - 32 * w;
    if (sh >= 0 && sh < 32) v |= wd[w] >> sh;
    if (sh < 0 && sh > -width) v |= wd[w] << (-sh);
  }
  return v & ((1u << width) - 1u);
}
template <int N>
__device__ __forceinline__ void set_bits_rt(uint32_t (&wd)[N], int pos, int width, uint32_t code) {
  const uint32_t m = (1u << width) - 1u;
#pragma unroll
  for (int w = 0; w < N; ++w) {
    const int sh = pos - 32 * w;
    if (sh >= 0 && sh < 32) wd[w] = (wd[w] & ~(m << sh)) | (code << sh);
    if (sh < 0 && sh > -width) wd[w] = (wd[w] & ~(m >> (-sh))) | (code >> (-sh));
  }
}

// Code of coordinate `col` (a run-time index) in a chunk's BM packed words, and its replacement.
template <int BM>
__device__ __forceinline__ uint32_t code_at(const uint32_t (&wd)[BM], int col) {
  const int pos = col * BM;
  uint32_t v = 0;
#pragma unroll
  for (int w = 0; w < BM; ++w) {
    const int sh = pos - 32 * w;
    if (sh >= 0 && sh < 32) v |= wd[w] >> sh;
    if (sh < 0 && sh > -BM) v |= wd[w] << (-sh);
  }
  return v & ((1u << BM) - 1u);
}
template <int BM>
__device__ __forceinline__ void set_code(uint32_t (&wd)[BM], int col, uint32_t code) {
  const int pos = col * BM;
  const uint32_t m = (1u << BM) - 1u;
#pragma unroll
  for (int w = 0; w < BM; ++w) {
    const int sh = pos - 32 * w;
    if (sh >= 0 && sh < 32) wd[w] = (wd[w] & ~(m << sh)) | (code << sh);
    if (sh < 0 && sh > -BM) wd[w] = (wd[w] & ~(m >> (-sh))) | (code >> (-sh));
  }
}

// A flagged coordinate redone exactly, by the whole warp: v = √d·⟨x_row, Π_col⟩/s
// as a float-float dot product (products split by an FMA, two-sum
// reduction).  Rare, so kept out of line: its temporaries then do not compete
// for the epilogue's registers.
template <bool F16>
__device__ __noinline__ float exact_coord(const void* x, const float* pi, double sqrt_d, int64_t row, int col,
                                          float s, int lane) {
  float4 xv;
  if constexpr (F16) {
    const uint2 h = __ldg(reinterpret_cast<const uint2*>(static_cast<const __half*>(x) + row * kDim) + lane);
    const float2 x0 = __half22float2(*reinterpret_cast<const __half2*>(&h.x));
    const float2 x1 = __half22float2(*reinterpret_cast<const __half2*>(&h.y));
    xv = make_float4(x0.x, x0.y, x1.x, x1.y);
  } else {
    xv = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(x) + row * kDim) + lane);
  }
  const float4 pv = __ldg(reinterpret_cast<const float4*>(pi + (int64_t)col * kDim) + lane);
  float sh = 0.f, sl = 0.f;
  ff_fma(xv.x, pv.x, sh, sl);
  ff_fma(xv.y, pv.y, sh, sl);
  ff_fma(xv.z, pv.z, sh, sl);
  ff_fma(xv.w, pv.w, sh, sl);
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float oh = __shfl_xor_sync(kFull, sh, o), ol = __shfl_xor_sync(kFull, sl, o);
    const float s2 = sh + oh, bb = s2 - sh;
    sl = sl + ol + ((sh - (s2 - bb)) + (oh - bb));
    sh = s2;
  }
  return (float)(((double)sh + (double)sl) * (sqrt_d / (double)s));
}

// The three-pass product of a tensor-memory A operand (hi at a0, lo at a0 + 64
// columns, K = 128) with a B table (hi, lo planes per 64-wide K chunk) into acc:
// lo·Bhi, hi·Blo, then hi·Bhi.
__device__ __forceinline__ void mma3_ts(uint32_t acc, uint32_t a0, uint32_t btab, uint32_t idesc) {
#pragma unroll
  for (int pass = 0; pass < 3; ++pass)
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const uint32_t a = a0 + (pass == 0 ? 64u : 0u) + 8u * ks;
      const uint32_t plane = pass == 1 ? 1u : 0u;
      const uint64_t bd = umma_desc(btab + ((ks >> 2) * 2 + plane) * kUmmaPlaneBytes + (ks & 3) * 256, 128, 1024);
      umma_f16_ts(acc, a, bd, idesc, (pass | ks) != 0 ? 1u : 0u);
    }
}

template <int BM, bool PROD, bool F16, bool MIX, bool PAIRL>
__global__ void __launch_bounds__(kEncThreads, 1) encode128_kernel(const Enc128Params p,
                                                                 const __grid_constant__ CUtensorMap xmap) {
  using L = Lay<F16, PROD>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // 1024-byte aligned base: the swizzled stages and their descriptors need it
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  unsigned char* sPi = smem;
  unsigned char* sM = smem + kTab;
  unsigned char* sX = smem + L::OffX;
  float* norm_s = reinterpret_cast<float*>(smem + L::OffNorm);  // [AccBufs][128]
  float* thr_s = reinterpret_cast<float*>(smem + L::OffThr);    // thresholds, +inf padded to 16
  float* cen_s = reinterpret_cast<float*>(smem + L::OffCen);    // centroids (MIX: the (BM+1)-bit thresholds)
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::OffBar);
  uint64_t* x_full = bars;         // [3] TMA bytes
  uint64_t* x_empty = bars + 3;    // [3] prep warps (+ the MMA commit for fp16 rows)
  uint64_t* a_full = bars + 6;     // [2] prep warps
  uint64_t* a_empty = bars + 8;    // [2] MMA commit
  uint64_t* acc_full = bars + 10;  // [2] MMA commit
  uint64_t* acc_empty = bars + 12; // [2] epilogue warps
  uint64_t* nb_full = bars + 14;   // [2] prep warps: the tile's norms are in norm_s
  uint64_t* nb_empty = bars + 16;  // [2] epilogue warps
  uint64_t* a2_full = bars + 18;   // Prod: epilogue warps wrote the residual operand
  uint64_t* a2_empty = bars + 19;  // MMA commit
  uint64_t* acc2_full = bars + 20; // MMA commit
  uint64_t* acc2_empty = bars + 21;// epilogue warps
  uint64_t* tab_full = bars + 22;  // the B tables
  uint64_t* drain = bars + 23;     // every MMA issued has completed
  uint64_t* g2_full = bars + 24;   // [2] Prod: both halves of the rows' γ² are in shared memory
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + L::NBar);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t ntiles = (p.N + kRows - 1) / kRows;
  const int nloc = ntiles > (int64_t)blockIdx.x ? (int)((ntiles - 1 - blockIdx.x) / gridDim.x + 1) : 0;
  const uint32_t lim = p.wait_limit;

  if (tid == 0) {
    for (int s = 0; s < L::XStages; ++s) {
      mbar_init(&x_full[s], 1);
      mbar_init(&x_empty[s], F16 ? 5 : 4);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&a_full[s], 4);
      mbar_init(&a_empty[s], 1);
      mbar_init(&acc_full[s], 1);
      mbar_init(&acc_empty[s], kEpiWarps);
      mbar_init(&nb_full[s], 4);
      mbar_init(&nb_empty[s], kEpiWarps);
      mbar_init(&g2_full[s], kEpiWarps);
    }
    mbar_init(a2_full, kEpiWarps);
    mbar_init(a2_empty, 1);
    mbar_init(acc2_full, 1);
    mbar_init(acc2_empty, kEpiWarps);
    mbar_init(tab_full, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (tid < 16) {
    thr_s[tid] = tid < (1 << BM) - 1 ? p.thr[tid] : INFINITY;
    if constexpr (MIX)
      cen_s[tid] = tid < (2 << BM) - 1 ? p.thr_hi[tid] : INFINITY;
    else
      cen_s[tid] = tid < (1 << BM) ? p.cen[tid] : 0.f;
  }
  if (warp == 0) tmem_alloc(tmem_slot, L::TmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------- producer
    uint32_t i = 0;
    if (lane == 0) {
      mbar_arrive_expect_tx(tab_full, (uint32_t)(kTab * (PROD ? 2 : 1)));
      bulk_g2s(sPi, p.tab_pi, kTab, tab_full);
      if (PROD) bulk_g2s(sM, p.tab_m, kTab, tab_full);
    }
    for (; (int)i < nloc; ++i) {
      const int64_t t = blockIdx.x + (int64_t)i * gridDim.x;
      const uint32_t s = i % L::XStages;
      if (!__all_sync(kFull, bar_wait(&x_empty[s], ((i / L::XStages) & 1u) ^ 1u, abort_flag, p.status, lim))) break;
      if (lane == 0) {
        // rows past N read as zeros and still count toward the box's bytes
        mbar_arrive_expect_tx(&x_full[s], (uint32_t)L::Stage);
#pragma unroll
        for (int bx = 0; bx < L::Boxes; ++bx)
          tma_load_2d(sX + s * L::Stage + bx * kBox, &xmap, bx * (128 / L::ES), (int)(t * kRows), &x_full[s]);
      }
      __syncwarp();
    }
    if (lane == 0) {
      // every copy this CTA issued lands before it may exit (bounded)
      const uint32_t first = i >= (uint32_t)L::XStages ? i - L::XStages : 0u;
      for (uint32_t j = first; j < i; ++j)
        for (uint32_t n = 0; n < kSpinLimitDev && !mbar_try_wait(&x_full[j % L::XStages], (j / L::XStages) & 1u); ++n) {
        }
      for (uint32_t n = 0; n < kSpinLimitDev && !mbar_try_wait(tab_full, 0u); ++n) {
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = umma_idesc_f16(kRows, kDim);
      const uint32_t bpi = smem_u32(sPi), bm = smem_u32(sM);
      bool ok = bar_wait(tab_full, 0u, abort_flag, p.status, lim);
      for (int i = 0; ok && i <= nloc; ++i) {
        if (i < nloc) {
          const uint32_t ab = i % L::AccBufs;
          if (!bar_wait(&acc_empty[ab], ((i / L::AccBufs) & 1u) ^ 1u, abort_flag, p.status, lim)) break;
          const uint32_t acc = tmem + L::ColAcc + ab * 128;
          if constexpr (F16) {
            const uint32_t s = i % L::XStages;
            if (!bar_wait(&x_full[s], (i / L::XStages) & 1u, abort_flag, p.status, lim)) break;
            tc_fence_after();
            const uint32_t xa = smem_u32(sX + s * L::Stage);
#pragma unroll
            for (int pass = 0; pass < 2; ++pass)  // x·Πlo, then x·Πhi
#pragma unroll
              for (int ks = 0; ks < 8; ++ks) {
                const uint64_t ad = umma_desc_sw128(xa + (ks >> 2) * kBox + (ks & 3) * 32);
                const uint64_t bd = umma_desc(
                    bpi + ((ks >> 2) * 2 + (pass == 0 ? 1 : 0)) * kUmmaPlaneBytes + (ks & 3) * 256, 128, 1024);
                umma_f16(acc, ad, bd, idesc, (pass | ks) != 0 ? 1u : 0u);
              }
            umma_commit(&x_empty[s]);
          } else {
            const uint32_t as = i % L::AStages;
            if (!bar_wait(&a_full[as], (i / L::AStages) & 1u, abort_flag, p.status, lim)) break;
            tc_fence_after();
            mma3_ts(acc, tmem + as * 128, bpi, idesc);
            umma_commit(&a_empty[as]);
          }
          umma_commit(&acc_full[ab]);
        }
        if (PROD && i >= 1) {  // the QJL product of the previous tile
          const uint32_t ph = (uint32_t)(i - 1) & 1u;
          if (!bar_wait(a2_full, ph, abort_flag, p.status, lim) ||
              !bar_wait(acc2_empty, ph ^ 1u, abort_flag, p.status, lim))
            break;
          tc_fence_after();
          mma3_ts(tmem + L::ColAcc2, tmem + L::ColA2, bm, idesc);
          umma_commit(a2_empty);
          umma_commit(acc2_full);
        }
      }
      // every MMA issued completes before tensor memory is released (bounded)
      umma_commit(drain);
      for (uint32_t n = 0; n < kSpinLimitDev && !mbar_try_wait(drain, 0u); ++n) {
      }
    }
  } else if (warp < 6) {
    // ---------------- prep: norms (and the split A operand of fp32 rows)
    const int q = warp & 3, r = 32 * q + lane, sw = r & 7;
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;
    for (int i = 0; i < nloc; ++i) {
      const uint32_t s = i % L::XStages;
      if (!__all_sync(kFull, bar_wait(&x_full[s], (i / L::XStages) & 1u, abort_flag, p.status, lim))) break;
      // 16-byte chunk c of row r of a box sits at chunk c ^ (r % 8) of its 128-byte row
      const unsigned char* row = sX + s * L::Stage + r * 128;
      float ss = 0.f;
      if constexpr (F16) {
#pragma unroll
        for (int bx = 0; bx < 2; ++bx)
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint4 u = *reinterpret_cast<const uint4*>(row + bx * kBox + 16 * (c ^ sw));
            const __half2* h = reinterpret_cast<const __half2*>(&u);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 f2 = __half22float2(h[e]);
              ss = fmaf(f2.x, f2.x, fmaf(f2.y, f2.y, ss));
            }
          }
      } else {
        // fp32 rows: one box per trip (the prep code shares each SMSP's
        // instruction cache with the epilogue's)
#pragma unroll 1
        for (int bx = 0; bx < 4; ++bx)
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const float4 f4 = *reinterpret_cast<const float4*>(row + bx * kBox + 16 * (c ^ sw));
            ss = fmaf(f4.x, f4.x, fmaf(f4.y, f4.y, fmaf(f4.z, f4.z, fmaf(f4.w, f4.w, ss))));
          }
      }
      float nrm = sqrtf(ss);
      if (!(ss > 1e-30f && ss < 1e36f)) {
        // squares near or past the ends of the fp32 range (or a zero row): sum
        // again with the row scaled by the power of two that brings its
        // largest magnitude to [1, 2)
        float m = 0.f;
#pragma unroll 1
        for (int k = 0; k < kDim; ++k) {
          const unsigned char* at = row + (k * L::ES / 128) * kBox + 16 * (((k * L::ES % 128) / 16) ^ sw) + (k * L::ES % 16);
          const float xv = F16 ? __half2float(*reinterpret_cast<const __half*>(at)) : *reinterpret_cast<const float*>(at);
          m = fmaxf(m, fabsf(xv));
        }
        nrm = 0.f;
        if (m > 0.f) {
          int e;
          frexpf(m, &e);
          const float scl = ldexpf(1.f, 1 - e);
          float s2 = 0.f;
#pragma unroll 1
          for (int k = 0; k < kDim; ++k) {
            const unsigned char* at = row + (k * L::ES / 128) * kBox + 16 * (((k * L::ES % 128) / 16) ^ sw) + (k * L::ES % 16);
            const float xv = (F16 ? __half2float(*reinterpret_cast<const __half*>(at)) : *reinterpret_cast<const float*>(at)) * scl;
            s2 = fmaf(xv, xv, s2);
          }
          nrm = sqrtf(s2) / scl;
        }
      }
      if constexpr (F16) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&x_empty[s]);
      }
      // the tile's norms to the epilogue
      const uint32_t ab = i % L::AccBufs;
      if (!__all_sync(kFull, bar_wait(&nb_empty[ab], ((i / L::AccBufs) & 1u) ^ 1u, abort_flag, p.status, lim))) break;
      norm_s[ab * kRows + r] = nrm;
      __syncwarp();
      if (lane == 0) mbar_arrive(&nb_full[ab]);
      if constexpr (!F16) {
        // A = x·2^e as fp16 hi + lo: hi plane columns [0, 64), lo plane [64, 128)
        // of the stage, column c holding coordinates 2c and 2c + 1
        const float sc = pow2_scale_16_32(nrm);
        const uint32_t as = i % L::AStages;
        if (!__all_sync(kFull, bar_wait(&a_empty[as], ((i / L::AStages) & 1u) ^ 1u, abort_flag, p.status, lim))) break;
        tc_fence_after();
#pragma unroll 1
        for (int bx = 0; bx < 4; ++bx) {  // 32 coordinates per box
          uint32_t hi[16], lo[16];
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const float4 f4 = *reinterpret_cast<const float4*>(row + bx * kBox + 16 * (c ^ sw));
            split2(f4.x * sc, f4.y * sc, hi[2 * c], lo[2 * c]);
            split2(f4.z * sc, f4.w * sc, hi[2 * c + 1], lo[2 * c + 1]);
          }
          tmem_st16(tmem + lane_base + as * 128 + 16 * bx, hi);
          tmem_st16(tmem + lane_base + as * 128 + 64 + 16 * bx, lo);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&a_full[as]);
          mbar_arrive(&x_empty[s]);
        }
      }
    }
  } else {
    // ---------------- epilogue: warps 6..; warp w serves TMEM lanes 32·(w % 4)..+31
    // (rows of the tile) and chunk c0 = (w - 6) / 4 of the four 32-column chunks
    const int q = warp & 3, r = 32 * q + lane, c0 = (warp - 6) >> 2;
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;
    const bool even = (lane & 1) == 0;
    for (int i = 0; i < nloc; ++i) {
      const int64_t t = blockIdx.x + (int64_t)i * gridDim.x;
      const int64_t row = t * kRows + r;
      const bool valid = row < p.N;
      const uint32_t ab = i % L::AccBufs, par = (i / L::AccBufs) & 1u;
      if (!__all_sync(kFull, bar_wait(&nb_full[ab], par, abort_flag, p.status, lim))) break;
      const float s = norm_s[ab * kRows + r];
      __syncwarp();
      if (lane == 0) mbar_arrive(&nb_empty[ab]);
      const float sc = F16 ? 1.f : pow2_scale_16_32(s);
      // fp32 on purpose: its rounding (~2e-7 relative) lies far inside the
      // recomputation band, and fp64 arithmetic is slow on this part
      const float f = s > 0.f ? p.sqrt_df / (s * sc * p.pi_scale) : 0.f;
      const bool live = valid && s > 0.f;
      // plain MSE and b + 1/2 bits compare the accumulator itself with the
      // thresholds divided by the row's scale 1/f, and the band with kMargin/f
      const float inv = s * sc * p.pi_scale / p.sqrt_df;
      const float mg = kMargin * inv;
      const int64_t dv = valid ? dest_row(p, row) : 0;
      if (!__all_sync(kFull, bar_wait(&acc_full[ab], par, abort_flag, p.status, lim))) break;
      tc_fence_after();
      const uint32_t acc = tmem + lane_base + L::ColAcc + ab * 128;
      // b = 4 plain MSE: eight columns per trip of a rolled loop (the unrolled
      // 32-column bucketize overflows the instruction cache at 7 thresholds)
      constexpr bool kGroups = !PROD && !MIX && !PAIRL && BM == 4;
      constexpr bool kMixHalves = MIX && BM == 3;  // 3.5 bits: two rolled halves of 16 columns
      uint32_t a0[(kGroups || kMixHalves) ? 1 : 32];
      if constexpr (!kGroups && !kMixHalves) {
        tmem_ld32_nw(acc + 32 * c0, a0);
        tmem_wait_ld();
      }
      // a3/a4 on the warp's 32-coordinate chunk c0: bucketize, flag, pack
      // (MSE and Prod: BM words, words [c0·BM, c0·BM + BM) of the row's
      // stream; b + 1/2 bits: 2·BM + 1 halfwords from halfword c0·(2·BM + 1)),
      // recompute flagged coordinates, store
      constexpr int HW = 2 * BM + 1;  // b + 1/2 bits: halfwords of a chunk
      uint32_t cw[BM];
      uint32_t hw[MIX ? BM + 1 : 1];  // b + 1/2 bits: the chunk's codes at mixed_pos
      uint32_t plo[PAIRL ? BM : 1], phi[PAIRL ? BM : 1];  // MSE, PAIR: slots of the pair block
#pragma unroll
      for (int w = 0; w < (MIX ? BM + 1 : 1); ++w) hw[w] = 0u;
      float g2 = 0.f;
      uint32_t m32;
      if constexpr (kMixHalves) {
        bool flagged = false;
        float tlo[kTB<BM>], thi[kTB<BM + 1>];
        scaled_thresholds<BM>(p.thr, inv, tlo);
        scaled_thresholds<BM + 1>(p.thr_hi, inv, thi);
        float dmin = INFINITY;
        constexpr int HB = 8 * (2 * BM + 1);  // bits of a half
#pragma unroll 1
        for (int g = 0; g < 2; ++g) {
          uint32_t a16[16];
          tmem_ld16_nw(acc + 32 * c0 + 16 * g, a16);
          tmem_wait_ld();
          const uint64_t cv = mix_half_codes<BM>(a16, tlo, thi, dmin);
          if (g == 0) {
            hw[0] |= (uint32_t)cv;
            hw[1] |= (uint32_t)(cv >> 32);
          } else {  // bits HB .. 2·HB of the chunk
#pragma unroll
            for (int w = 0; w <= BM; ++w) {
              const int lo = 32 * w - HB;  // bit of cv at the start of word w
              uint32_t x = 0u;
              if (lo >= 0 && lo < 64) x = (uint32_t)(cv >> lo);
              if (lo < 0 && lo > -32) x = (uint32_t)(cv << (-lo));
              hw[w] |= x;
            }
          }
        }
        flagged = dmin < mg;
        m32 = 0u;
        if (__any_sync(kFull, flagged && live)) {  // rare: the flags, from tensor memory again
          uint32_t t32[32];
          tmem_ld32_nw(acc + 32 * c0, t32);
          tmem_wait_ld();
          if (flagged) m32 = mix_near_mask<BM>(t32, f, p.thr, p.thr_hi);
        }
      } else if constexpr (MIX) {
        bool flagged = false;
        float tlo[kTB<BM>], thi[kTB<BM + 1>];
        scaled_thresholds<BM>(p.thr, inv, tlo);
        scaled_thresholds<BM + 1>(p.thr_hi, inv, thi);
        mix_chunk_codes<BM>(a0, tlo, thi, mg, hw, flagged);
        m32 = 0u;
        if (__any_sync(kFull, flagged && live)) {  // rare: the flags, from tensor memory again
          uint32_t t32[32];
          tmem_ld32_nw(acc + 32 * c0, t32);
          tmem_wait_ld();
          if (flagged) m32 = mix_near_mask<BM>(t32, f, p.thr, p.thr_hi);
        }
      } else if constexpr (PAIRL) {
        bool flagged = false;
        float tb[kTB<BM>];
        scaled_thresholds<BM>(p.thr, inv, tb);
        chunk_codes_pair<BM>(a0, tb, mg, plo, phi, flagged);
        m32 = 0u;
        if (__any_sync(kFull, flagged && live)) {
          uint32_t t32[32];
          tmem_ld32_nw(acc + 32 * c0, t32);
          tmem_wait_ld();
          if (flagged) m32 = near_mask<BM>(t32, f, p.thr);
        }
      } else {
        bool flagged = false;
        if constexpr (kGroups) {
          float tb[kTB<BM>];
          scaled_thresholds<BM>(p.thr, inv, tb);
          float dmin = INFINITY;
#pragma unroll
          for (int w = 0; w < BM; ++w) cw[w] = 0u;
#pragma unroll 1
          for (int k = 0; k < 4; ++k) {
            uint32_t a8[8];
            tmem_ld8_nw(acc + 32 * c0 + 8 * k, a8);
            tmem_wait_ld();
            uint32_t wd = 0u;
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) wd |= bucketize_sc<BM>(__uint_as_float(a8[jj]), tb, dmin) << (4 * jj);
#pragma unroll
            for (int w = 0; w < BM; ++w) cw[w] = w == k ? wd : cw[w];
          }
          flagged = dmin < mg;
          m32 = 0u;
        } else if constexpr (!PROD) {
          float tb[kTB<BM>];
          scaled_thresholds<BM>(p.thr, inv, tb);
          chunk_codes_s<BM>(a0, tb, mg, cw, flagged);
          m32 = 0u;
        } else {
          prod_chunk_codes<BM>(a0, f, p.thr, cen_s, cw, g2, flagged);
          m32 = 0u;
        }
        // a chunk with a coordinate near a threshold (~1e-3 of them): its
        // values again from tensor memory (not yet handed back), then the flags
        if (__any_sync(kFull, flagged && live)) {
          uint32_t t32[32];
          tmem_ld32_nw(acc + 32 * c0, t32);
          tmem_wait_ld();
          if (flagged) m32 = near_mask<BM>(t32, f, p.thr);
        }
      }
      // the accumulator goes back to the MMA (the kernel is epilogue-bound,
      // so the MMA loses nothing by waiting for a flagged chunk's re-read)
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[ab]);
      if (!live) {
#pragma unroll
        for (int w = 0; w < BM; ++w) cw[w] = 0u;
#pragma unroll
        for (int w = 0; w < (MIX ? BM + 1 : 1); ++w) hw[w] = 0u;
#pragma unroll
        for (int w = 0; w < (PAIRL ? BM : 1); ++w) plo[w] = phi[w] = 0u;
        m32 = 0u;
        g2 = 0.f;
      }
      // flagged coordinates: one warp-wide float-float dot product each
      for (;;) {
        const uint32_t any = __ballot_sync(kFull, m32 != 0u);
        if (!any) break;
        const int src = __ffs(any) - 1;
        int j = 0;
        if (lane == src) {
          j = __ffs(m32) - 1;
          m32 &= m32 - 1u;
        }
        j = __shfl_sync(kFull, j, src);
        const float ssrc = __shfl_sync(kFull, s, src);
        const float vv = exact_coord<F16>(p.x, p.pi, p.sqrt_d, t * kRows + 32 * q + src, 32 * c0 + j, ssrc, lane);
        if (lane == src) {
          bool nr;
          if constexpr (MIX) {
            const bool hi = (j & 8) == 0;
            const uint32_t code = hi ? bucketize<BM + 1>(vv, cen_s, 0.f, nr) : bucketize<BM>(vv, thr_s, 0.f, nr);
            set_bits_rt(hw, mixed_pos(j, BM), hi ? BM + 1 : BM, code);
          } else if constexpr (PAIRL) {
            const uint32_t code = bucketize<BM>(vv, thr_s, 0.f, nr);
            if (j < 16)
              set_bits_rt(plo, 2 * j * BM, BM, code);
            else
              set_bits_rt(phi, 2 * (j - 16) * BM, BM, code);
          } else {
            const uint32_t code = bucketize<BM>(vv, thr_s, 0.f, nr);
            if constexpr (PROD) {
              const uint32_t old = code_at<BM>(cw, j);
              const float e0 = vv - cen_s[old], e1 = vv - cen_s[code];
              g2 += e1 * e1 - e0 * e0;
            }
            set_code<BM>(cw, j, code);
          }
        }
      }
      // stores of the chunk's codes
      if constexpr (PAIRL) {
        // PAIR (vectors 2k and 2k+1 share a block; coordinate j's two codes
        // side by side at block bits 2j·BM, even vector low): the chunk's
        // block is 2·BM words from word 2·c0·BM; lo holds its first BM words'
        // fields of this vector, hi the last BM.  When the destination pairs
        // rows r and r+1 (lanes l and l+1), the even lane writes the first BM
        // words and the odd lane the rest, after one exchange.
        const bool odd = (dv & 1) != 0;
        if (odd) {
          shift_slot<BM>(plo);
          shift_slot<BM>(phi);
        }
        const int64_t base_row = row - (even ? 0 : 1);
        const bool whole = p.pair_aligned && base_row + 1 < p.N;
        uint32_t* blk = p.codes + (dv >> 1) * (2 * (int64_t)p.W) + 2 * c0 * BM;
        uint32_t ow[BM];
#pragma unroll
        for (int w = 0; w < BM; ++w) ow[w] = (even ? plo[w] : phi[w]) | __shfl_xor_sync(kFull, even ? phi[w] : plo[w], 1);
        if (valid && whole) {
          store_words<BM>(blk + (even ? 0 : BM), ow);
        } else if (valid) {
          // the partner is written by another call (or not at all): this
          // vector's slots of the 2·BM block words by masked atomics
          uint32_t m0[BM];
#pragma unroll
          for (int w = 0; w < BM; ++w) m0[w] = 0u;
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) put_bits<BM>(m0, 2 * jj * BM, (1u << BM) - 1u);
          if (odd) shift_slot<BM>(m0);
#pragma unroll
          for (int w = 0; w < BM; ++w) {
            atomicAnd(blk + w, ~m0[w]);
            atomicOr(blk + w, plo[w]);
            atomicAnd(blk + BM + w, ~m0[w]);
            atomicOr(blk + BM + w, phi[w]);
          }
        }
      } else if constexpr (MIX) {
        if (p.layout == TQ_LAYOUT_TOKEN) {
          if (valid) {
            store_halfwords<BM>(reinterpret_cast<uint16_t*>(p.codes + dv * p.W) + c0 * HW, hw);
          }
        } else {
          // PAIR: coordinate j's field of 2·w_j bits at block bit 2·P_j; the
          // chunk's block is 2·HW halfwords from halfword 2·c0·HW.  Rows r and
          // r+1 of the tile are lanes l and l+1; when the destination pairs them,
          // the even lane writes the fields of coordinates 0-15 (halfwords
          // [0, HW)), the odd lane those of 16-31 ([HW, 2·HW), the same offsets
          // within), after one exchange.
          uint32_t part[BM + 1];
#pragma unroll
          for (int w = 0; w <= BM; ++w) part[w] = __shfl_xor_sync(kFull, hw[w], 1);
          const int64_t base_row = row - (even ? 0 : 1);
          const bool whole = p.pair_aligned && base_row + 1 < p.N;
          uint32_t* blk = p.codes + (dv >> 1) * (2 * (int64_t)p.W) + c0 * HW;
          if (valid && whole) {
            // the even and odd vectors' codes of this lane's 16 coordinates
            // (the odd lane's start 8·HW bits into the chunk)
            constexpr int K = 8 * HW;
            uint32_t E[BM + 1], O[BM + 1], ev[BM + 1], od[BM + 1], ob[BM + 1];
#pragma unroll
            for (int w = 0; w <= BM; ++w) {
              E[w] = even ? hw[w] : part[w];
              O[w] = even ? part[w] : hw[w];
            }
#pragma unroll
            for (int w = 0; w <= BM; ++w) {
              const int lo = (K + 32 * w) >> 5, sh = (K + 32 * w) & 31;
              uint32_t se = 0u, so = 0u;
              if (lo <= BM) {
                se = E[lo] >> sh;
                so = O[lo] >> sh;
              }
              if (sh != 0 && lo + 1 <= BM) {
                se |= E[lo + 1] << (32 - sh);
                so |= O[lo + 1] << (32 - sh);
              }
              ev[w] = even ? E[w] : se;
              od[w] = even ? O[w] : so;
              ob[w] = 0u;
            }
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              const int pk = mixed_pos(k, BM);
              if ((k & 8) == 0) {
                put_bits<BM + 1>(ob, 2 * pk, get_bits<BM + 1>(ev, pk));
                put_bits<BM + 1>(ob, 2 * pk + BM + 1, get_bits<BM + 1>(od, pk));
              } else {
                put_bits<BM>(ob, 2 * pk, get_bits<BM>(ev, pk));
                put_bits<BM>(ob, 2 * pk + BM, get_bits<BM>(od, pk));
              }
            }
            uint16_t* dst = reinterpret_cast<uint16_t*>(blk) + (even ? 0 : HW);
            store_halfwords<BM>(dst, ob);
          } else if (valid) {
            // the partner is written by another call (or not at all): this
            // vector's fields of the chunk's HW block words by masked atomics
            // (word by word: only the fields overlapping word w, a compile-time
            // test once both loops are unrolled; the slot picks the shift)
            const bool odd = (dv & 1) != 0;
            auto shift = [](uint32_t x, int sh) -> uint32_t {
              return sh >= 32 || sh <= -32 ? 0u : (sh >= 0 ? x << sh : x >> (-sh));
            };
#pragma unroll
            for (int w = 0; w < HW; ++w) {
              uint32_t fb = 0u, mb = 0u;
#pragma unroll
              for (int k = 0; k < 32; ++k) {
                const int wk = (k & 8) ? BM : BM + 1, pk = mixed_pos(k, BM);
                const int p0 = 2 * pk - 32 * w;  // the pair field of coordinate k, relative to word w
                if (p0 >= 32 || p0 + 2 * wk <= 0) continue;
                const int sh = odd ? p0 + wk : p0;
                fb |= shift(get_bits_rt(hw, pk, wk), sh);
                mb |= shift((1u << wk) - 1u, sh);
              }
              atomicAnd(blk + w, ~mb);
              atomicOr(blk + w, fb);
            }
          }
        }
      } else if (p.layout == TQ_LAYOUT_TOKEN) {
        if (valid) {
          uint32_t* dst = p.codes + dv * p.W + c0 * BM;
          if constexpr (BM == 3) {  // three word stores measured faster here than 8 + 4 bytes
#pragma unroll
            for (int w = 0; w < BM; ++w) dst[w] = cw[w];
          } else {
            store_words<BM>(dst, cw);
          }
        }
      } else {
        // PAIR: vectors 2k and 2k+1 share a block; coordinate j's two codes
        // sit side by side at block bits 2j·BM (even vector low).  Rows r and
        // r+1 of the tile are lanes l and l+1; when the destination pairs them,
        // the even lane writes the block words of coordinates 32c..32c+15 and
        // the odd lane those of 32c+16..32c+31, after one exchange.
        uint32_t part[BM];
#pragma unroll
        for (int w = 0; w < BM; ++w) part[w] = __shfl_xor_sync(kFull, cw[w], 1);
        const int64_t base_row = row - (even ? 0 : 1);
        const bool whole = p.pair_aligned && base_row + 1 < p.N;
        uint32_t* blk = p.codes + (dv >> 1) * (2 * (int64_t)p.W) + 2 * c0 * BM;
        if (valid && whole) {
          uint32_t ow[BM];
#pragma unroll
          for (int w = 0; w < BM; ++w) ow[w] = 0u;
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            const uint32_t own = even ? get_bits<BM>(cw, jj * BM) : get_bits<BM>(cw, (16 + jj) * BM);
            const uint32_t prt = even ? get_bits<BM>(part, jj * BM) : get_bits<BM>(part, (16 + jj) * BM);
            put_bits<BM>(ow, 2 * jj * BM, even ? own : prt);
            put_bits<BM>(ow, (2 * jj + 1) * BM, even ? prt : own);
          }
          store_words<BM>(blk + (even ? 0 : BM), ow);
        } else if (valid) {
          // the partner is written by another call (or not at all): this
          // vector's fields of the chunk's 2·BM block words by masked atomics
          // (both slots built at compile-time positions, then picked)
          const bool odd = (dv & 1) != 0;
          uint32_t f0[2 * BM], f1[2 * BM], m0[2 * BM], m1[2 * BM];
#pragma unroll
          for (int w = 0; w < 2 * BM; ++w) f0[w] = f1[w] = m0[w] = m1[w] = 0u;
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) {
            const uint32_t code = get_bits<BM>(cw, jj * BM);
            put_bits<BM>(f0, 2 * jj * BM, code);
            put_bits<BM>(f1, (2 * jj + 1) * BM, code);
            put_bits<BM>(m0, 2 * jj * BM, (1u << BM) - 1u);
            put_bits<BM>(m1, (2 * jj + 1) * BM, (1u << BM) - 1u);
          }
#pragma unroll
          for (int w = 0; w < 2 * BM; ++w) {
            atomicAnd(blk + w, ~(odd ? m1[w] : m0[w]));
            atomicOr(blk + w, odd ? f1[w] : f0[w]);
          }
        }
      }
      if (valid && c0 == 0) p.norm[dv] = s;
      // a5 (Prod): γ over the row's four chunks, this chunk's residual operand,
      // the second product, this chunk's signs
      if constexpr (PROD) {
        float* g2_s = norm_s + L::AccBufs * kRows;  // [2 tile parities][4 chunks][128]
        g2_s[((i & 1) * 4 + c0) * kRows + r] = g2;
        __syncwarp();
        if (lane == 0) mbar_arrive(&g2_full[i & 1]);
        if (!__all_sync(kFull, bar_wait(&g2_full[i & 1], ((uint32_t)i >> 1) & 1u, abort_flag, p.status, lim))) break;
        const float* g2r = g2_s + (i & 1) * 4 * kRows + r;
        const float g2t = (g2r[0] + g2r[kRows]) + (g2r[2 * kRows] + g2r[3 * kRows]);
        const float gam = live ? sqrtf(fmaxf(g2t, 0.f)) / (float)p.sqrt_d : 0.f;
        const float rsd = live ? pow2_scale_16_32(gam) / (float)p.sqrt_d : 0.f;
        if (!__all_sync(kFull, bar_wait(a2_empty, ((uint32_t)i & 1u) ^ 1u, abort_flag, p.status, lim))) break;
        tc_fence_after();
        const uint32_t a2 = tmem + lane_base + L::ColA2;
        // two halves of 16 columns (8 packed words each), so that the
        // temporaries of the split stay within the register budget
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t hi[8], lo[8];
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            const int j = 8 * hf + jj;
            const float r0 = (__uint_as_float(a0[2 * j]) * f - cen_s[get_bits<BM>(cw, 2 * j * BM)]) * rsd;
            const float r1 = (__uint_as_float(a0[2 * j + 1]) * f - cen_s[get_bits<BM>(cw, (2 * j + 1) * BM)]) * rsd;
            split2(r0, r1, hi[jj], lo[jj]);
          }
          tmem_st8(a2 + 16 * c0 + 8 * hf, hi);
          tmem_st8(a2 + 64 + 16 * c0 + 8 * hf, lo);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(a2_full);
        if (!__all_sync(kFull, bar_wait(acc2_full, (uint32_t)i & 1u, abort_flag, p.status, lim))) break;
        tc_fence_after();
        uint32_t bits = 0u;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t pa[16];
          tmem_ld16_nw(tmem + lane_base + L::ColAcc2 + 32 * c0 + 16 * hf, pa);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 16; ++j) bits |= (__uint_as_float(pa[j]) >= 0.f ? 1u : 0u) << (16 * hf + j);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acc2_empty);
        if (valid) {
          p.qjl[dv * p.QW + c0] = live ? bits : 0u;
          if (c0 == 0) p.rnorm[dv] = gam;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, L::TmemCols);
  }
}

template <int BM, bool PROD, bool F16, bool MIX = false, bool PAIRL = false>
cudaError_t launch_t(const Enc128Params& p, const CUtensorMap& xmap, cudaStream_t st) {
  auto k = encode128_kernel<BM, PROD, F16, MIX, PAIRL>;
  static PerDeviceValue attr;  // set once per device, before any stream capture
  const cudaError_t e = smem_attr_once(attr, (const void*)k, Lay<F16, PROD>::SmemAlloc);
  if (e != cudaSuccess) return e;
  const int64_t tiles = (p.N + kRows - 1) / kRows;
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(tiles, (int64_t)num_sms()));
  k<<<grid, kEncThreads, Lay<F16, PROD>::SmemAlloc, st>>>(p, xmap);
  return cudaGetLastError();
}

template <bool F16>
cudaError_t launch_mode(const Enc128Params& p, const CUtensorMap& xmap, int bm, bool prod, bool mix,
                        cudaStream_t st) {
  if (mix) {
    switch (bm) {
      case 1: return launch_t<1, false, F16, true>(p, xmap, st);
      case 2: return launch_t<2, false, F16, true>(p, xmap, st);
      case 3: return launch_t<3, false, F16, true>(p, xmap, st);
    }
    return cudaErrorInvalidValue;
  }
  if (prod) {
    switch (bm) {
      case 1: return launch_t<1, true, F16>(p, xmap, st);
      case 2: return launch_t<2, true, F16>(p, xmap, st);
      case 3: return launch_t<3, true, F16>(p, xmap, st);
    }
    return cudaErrorInvalidValue;
  }
  if (p.layout == TQ_LAYOUT_PAIR) {  // plain MSE into PAIR caches: its own kernel
    switch (bm) {
      case 1: return launch_t<1, false, F16, false, true>(p, xmap, st);
      case 2: return launch_t<2, false, F16, false, true>(p, xmap, st);
      case 3: return launch_t<3, false, F16, false, true>(p, xmap, st);
      case 4: return launch_t<4, false, F16, false, true>(p, xmap, st);
    }
    return cudaErrorInvalidValue;
  }
  switch (bm) {
    case 1: return launch_t<1, false, F16>(p, xmap, st);
    case 2: return launch_t<2, false, F16>(p, xmap, st);
    case 3: return launch_t<3, false, F16>(p, xmap, st);
    case 4: return launch_t<4, false, F16>(p, xmap, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

bool enc128_supported(const DevCtx& c) {
  // symmetric codebooks only (tq_codebook_build makes them; the bucketize
  // compares |v| with the positive thresholds); others take the general encoder
  return c.d == kDim && c.enc_tab != nullptr && (c.mode != TQ_PROD || c.enc_tab_m != nullptr) &&
         c.b_mse >= 1 && c.b_mse <= (c.mode == TQ_MSE ? 4 : 3) && c.sym_thr != 0;
}

tq_status launch_encode128(const DevCtx& c, const void* x, int x_dtype, int64_t N, const tq_codes* out,
                           int64_t offset, int64_t group_rows, int64_t group_stride, cudaStream_t stream) {
  if (!enc128_supported(c)) return TQ_ERR_UNSUPPORTED;
  if (N > INT32_MAX) return TQ_ERR_UNSUPPORTED;  // TMA row coordinates are 32-bit
  Enc128Params p;
  p.x = x;
  p.N = N;
  p.codes = out->d_codes;
  p.norm = out->d_norm;
  p.qjl = out->d_qjl;
  p.rnorm = out->d_rnorm;
  p.tab_pi = c.enc_tab;
  p.tab_m = c.enc_tab_m;
  p.pi = c.pi;
  p.pi_scale = c.pi_scale;
  p.sqrt_d = std::sqrt((double)c.d);
  p.sqrt_df = (float)p.sqrt_d;
  for (int k = 0; k < 15; ++k) p.thr[k] = c.thr[k];
  for (int k = 0; k < 16; ++k) p.cen[k] = c.cen[k];
  for (int k = 0; k < 15; ++k) p.thr_hi[k] = c.thr_hi[k];
  const bool mix = c.mode == TQ_MIXED;
  p.layout = out->layout;
  p.W = c.words_per_vec;
  p.QW = c.qjl_words_per_vec;
  p.offset = offset;
  p.group_rows = group_rows;
  p.group_stride = group_stride;
  p.pair_aligned = (offset % 2 == 0) && (group_rows % 2 == 0 || group_rows >= N) && (group_stride % 2 == 0);
  p.status = c.status;
  p.wait_limit = c.wait_limit;
  CUtensorMap xmap;
  const tq_status ms = rows_tensor_map(&xmap, x, N, c.d, x_dtype == TQ_F16);
  if (ms != TQ_OK) return ms;
  const cudaError_t e = x_dtype == TQ_F16 ? launch_mode<true>(p, xmap, c.b_mse, c.mode == TQ_PROD, mix, stream)
                                          : launch_mode<false>(p, xmap, c.b_mse, c.mode == TQ_PROD, mix, stream);
  return e == cudaSuccess ? TQ_OK : set_cuda_error(e);
}

}  // namespace tq
