// Internal declarations shared by the host code and the kernels of libtq.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "tq.h"
#include "tq_once.h"

namespace tq {

// ------------------------------------------------------------------ limits
constexpr int kMaxD = 3072;
constexpr int kChunk = 128;       // output coordinates per encoder chunk
constexpr int kWarpRows = 16;     // rows (vectors) per warp tile of the encoder
constexpr int kEncWarps = 8;      // warps per encoder CTA

// Device-side view of a context, passed by value to kernels.
// tcgen05 encoder for d > 128: Π tiles of kUmmaTN outputs x kUmmaKC inputs, two fp16 planes each
constexpr int kUmmaTN = 128;
constexpr int kUmmaKC = 64;
constexpr int kUmmaPlaneBytes = kUmmaTN * kUmmaKC * 2;

// Polls a bounded pipeline wait makes before it gives up (tq_debug_set_wait_limit).
constexpr uint32_t kWaitLimitDefault = 1u << 22;

struct DevCtx {
  int d, b, b_mse, mode, rot;
  uint32_t wait_limit;   // polls of a bounded pipeline wait before it gives up
  int words_per_vec, qjl_words_per_vec;
  float sqrt_d;
  float pi_scale;        // encoder B operand = pi_scale * Π (power of two)
  float m_scale;         // QJL B operand = m_scale * S·Πᵀ (power of two)
  float alpha;           // LUT values are fp16(alpha * centroid)
  float thr[15];         // thresholds, unit-variance units (fp32)
  float cen[16];         // centroids, unit-variance units (fp32)
  float thr_hi[15];      // TQ_MIXED: the (b+1)-bit codebook's thresholds
  int sym_thr;           // thresholds (both sets for TQ_MIXED) symmetric about 0 in fp32
  float cen_hi[16];      // TQ_MIXED: the (b+1)-bit codebook's centroids
  const uint2* enc_pi;   // encoder B fragments of Π (hi/lo)
  const uint2* enc_m;    // encoder B fragments of S·Πᵀ (hi/lo), Prod only
  const float* pi;       // Π, d×d row-major fp32
  const float* s_mat;    // S, d×d row-major fp32, Prod only
  const float4* pi_slices;  // d = 128: Π[r][32c + 4j .. +3] at (c·8 + j)·128 + r (decode rotation)
  const float4* s_slices;   // d = 128, Prod: S in the same slices (decode S-rotation of the query)
  const unsigned char* umma_tab;  // d > 128, MSE: pi_scale·Π hi/lo tiles for the tcgen05 encoder (else null)
  const unsigned char* enc_tab;    // d = 128: pi_scale·Π hi/lo tiles for the tcgen05 encoder (else null)
  const unsigned char* enc_tab_m;  // d = 128, Prod: m_scale·S·Πᵀ in the same layout (else null)
  const float* signs;    // Hadamard rotation: σ, d entries of ±1 (else null)
  int had_m, had_p;      // Hadamard rotation: H = H12 ⊗ H_m (had_p = 12) or H_m (had_p = 1)
  const uint32_t* lut;   // pair table: 2^(2 b_mse) fp16x2 entries (alpha-scaled)
  const uint32_t* lut_hi;  // TQ_MIXED: pair table of the (b+1)-bit codebook, same alpha
  int* status;           // device status word
};

struct Ctx {
  DevCtx dev;
  tq_codebook cb;
  tq_codebook cb_hi;        // TQ_MIXED: the (b+1)-bit codebook
  double* h_pi = nullptr;   // d×d fp64
  double* h_s = nullptr;    // d×d fp64 (Prod)
  void* d_alloc = nullptr;  // single device allocation holding every table
  size_t d_bytes = 0;
};

tq_status set_cuda_error(cudaError_t e);

inline int words_per_vector(int d, int bits) {
  int w = (bits * d + 31) / 32;
  return (w + 3) / 4 * 4;
}

// b + 1/2 bits per coordinate: coordinate j has b + 1 bits where j mod 16 < 8,
// b elsewhere; its code starts at stream bit mixed_pos(j, b).  Every block of 16
// coordinates spans 8·(2b+1) bits, so d = 128 needs d·(2b+1)/64 whole words.
__host__ __device__ constexpr int mixed_width(int j, int b) { return (j & 8) ? b : b + 1; }
__host__ __device__ constexpr int mixed_pos(int j, int b) {
  return (j >> 4) * 8 * (2 * b + 1) + ((j & 8) ? 8 * (b + 1) + (j & 7) * b : (j & 7) * (b + 1));
}
inline int mixed_words_per_vector(int d, int b) { return d * (2 * b + 1) / 64; }

// kernel launchers (defined in the .cu files)
tq_status launch_encode(const DevCtx& c, const void* x, int x_dtype, int64_t N, const tq_codes* out,
                        int64_t offset, int64_t group_rows, int64_t group_stride,
                        cudaStream_t stream);
tq_status launch_scores(const DevCtx& c, const float* q, int M, const tq_codes* keys, int64_t first,
                        int64_t N, float* scores, void* ws, size_t ws_bytes, cudaStream_t stream);
size_t scores_ws_bytes(const DevCtx& c, int M);
tq_status launch_decode(const DevCtx& kc, const DevCtx& vc, const void* q, int q_dtype,
                        const tq_codes* K, const tq_codes* V, int B, int Hq, int Hkv, int64_t seq,
                        int64_t cap, float scale, float* out, void* ws, size_t ws_bytes,
                        cudaStream_t stream);
size_t decode_ws_bytes(int d, int B, int Hq, int Hkv, int64_t seq);
tq_status launch_decode_noalloc(const DevCtx& kc, const DevCtx& vc, const void* q, int q_dtype,
                                const tq_codes* K, const tq_codes* V, int B, int Hq, int Hkv,
                                int64_t seq, int64_t cap, float scale, float* out,
                                cudaStream_t stream);
size_t decode_noalloc_limit();
tq_status launch_step(const DevCtx& kc, const DevCtx& vc, const void* q, int q_dtype,
                      const void* knew, const void* vnew, int new_dtype, const tq_codes* K,
                      const tq_codes* V, int B, int Hq, int Hkv, int64_t seq, int64_t cap,
                      float scale, float* out, void* ws, cudaStream_t stream);
bool wht_supported(const DevCtx& c);
bool enc128_supported(const DevCtx& c);
tq_status launch_encode128(const DevCtx& c, const void* x, int x_dtype, int64_t N, const tq_codes* out,
                           int64_t offset, int64_t group_rows, int64_t group_stride, cudaStream_t stream);
// 2-D tensor map of N rows of d fp32/fp16 values for TMA loads of boxes of
// 128 rows x 128 bytes in the 128-byte swizzle.
tq_status rows_tensor_map(CUtensorMap* map, const void* x, int64_t N, int d, bool f16);
bool umma_supported(const DevCtx& c);
tq_status launch_encode_umma(const DevCtx& c, const void* x, int x_dtype, int64_t N, const tq_codes* out,
                             int64_t offset, int64_t group_rows, int64_t group_stride, cudaStream_t stream);
tq_status launch_encode_wht(const DevCtx& c, const void* x, int x_dtype, int64_t N, const tq_codes* out,
                            int64_t offset, int64_t group_rows, int64_t group_stride, cudaStream_t stream);
// SM count of the current device (cached per device).
int num_sms();
// Current device, or -1 if the runtime cannot tell.
int current_device();
// cudaFuncAttributeMaxDynamicSharedMemorySize = bytes for `func` on the current
// device, set once per device (`flag` is the kernel's own per-device record).
cudaError_t smem_attr_once(PerDeviceValue& flag, const void* func, int bytes);
// CTAs of `func` resident per SM with `threads` threads and `smem` bytes of
// dynamic shared memory, on the current device (cached per device in `cache`;
// 1 if the runtime cannot tell).
int ctas_per_sm_once(PerDeviceValue& cache, const void* func, int threads, size_t smem);
// One-time launch setup of the Hadamard fast transform for a context's shapes.
tq_status prime_encode_wht(const DevCtx& c);

}  // namespace tq
