/*
 * tq.h — C ABI of the TurboQuant hot path for NVIDIA GB300 (sm_103a).
 *
 * The method (TurboQuant, arXiv:2504.19874) as explained by the pages
 *   [P1] "TurboQuant 详解" (wnma3mz.github.io/hexo_blog, 2026-03-30)
 *   [P2] "turboquant-first-principles-walkthrough" (blog.hotdry.top, 2026-04-27)
 *   [P3] "压缩与速度的博弈——TurboQuant 和 RotorQuant 的真相" (zhichai.net)
 *   [P4] "sub-byte-kv-cache-quantization-turboquant" (blog2.hotdry.top, 2026-03-28)
 *
 * Conventions shared by every call
 * --------------------------------
 * - Pointers named d_* are DEVICE pointers owned by the caller (allocate them
 *   with any allocator, e.g. PyTorch).  Pointers named h_* are host pointers.
 *   The library allocates device memory only inside tq_ctx_create and frees it
 *   in tq_ctx_destroy.
 * - Every call that takes a stream is asynchronous on that stream, except
 *   where stated.  A NULL stream is the legacy default stream.
 * - Arguments are validated before anything is launched; on an error nothing
 *   has been written.  Errors: TQ_ERR_INVALID_ARG (bad value, NULL or
 *   misaligned pointer), TQ_ERR_UNSUPPORTED (valid but not implemented, e.g.
 *   a dimension outside the supported set), TQ_ERR_CUDA (a CUDA call failed;
 *   tq_last_cuda_error() gives the CUDA error code), TQ_ERR_ALLOC (device
 *   allocation in tq_ctx_create failed), TQ_ERR_TIMEOUT (a bounded device wait
 *   ran out; reported by tq_status_poll).
 * - Vector dimension d: a multiple of 32, at most 3072; d <= 128 or
 *   d % 128 == 0.  Bits b per coordinate: 1..4 (TurboQuant_Prod: 2..4).
 * - Units: codebooks are in "unit-variance units": a coordinate y_i of the
 *   rotated unit vector is compared as v_i = sqrt(d) * y_i.
 */
#ifndef TQ_H_
#define TQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* tq_stream; /* same type as cudaStream_t */

typedef enum {
  TQ_OK = 0,
  TQ_ERR_INVALID_ARG = -1,
  TQ_ERR_UNSUPPORTED = -2,
  TQ_ERR_CUDA = -3,
  TQ_ERR_ALLOC = -4,
  TQ_ERR_TIMEOUT = -5
} tq_status;

typedef enum { TQ_MSE = 0, TQ_PROD = 1, TQ_MIXED = 2 } tq_mode;
typedef enum { TQ_ROT_DENSE = 0, TQ_ROT_HADAMARD = 1 } tq_rot_kind;
typedef enum { TQ_DENS_BETA = 0, TQ_DENS_GAUSS = 1 } tq_density;
typedef enum { TQ_F32 = 0, TQ_F16 = 1 } tq_dtype;
typedef enum { TQ_LAYOUT_TOKEN = 0, TQ_LAYOUT_PAIR = 1 } tq_layout;

/* Library version string, e.g. "tq 0.1 sm_103a". */
const char* tq_version(void);

/* Human-readable name of a status code.  Never NULL. */
const char* tq_status_string(tq_status s);

/* CUDA error code (cudaError_t as int) of the last TQ_ERR_CUDA in this
 * process, 0 if none. */
int tq_last_cuda_error(void);

/* ------------------------------------------------------------------ codebook
 * Offline Lloyd-Max scalar quantizer for the coordinate density of a randomly
 * rotated unit vector.  [P1] section "痛点 2" (the two-step iteration: midpoint
 * thresholds, then cell means), section "关键洞察：先旋转" (the density
 * f_X(x) = Γ(d/2)/(√π Γ((d-1)/2)) (1-x²)^((d-3)/2), N(0,1/d) for large d);
 * [P4] section "工程实现的关键路径" (50 000-point grid over ±6σ, 300
 * iterations, computed once per (d, b) and cached).
 *
 * Host only, synchronous, pure (no device work).  grid <= 0 means 50000,
 * iters <= 0 means 300.  Initial centroids: the (k+1/2)/2^b quantiles of the
 * weighted grid's midpoint CDF; centroids are symmetrised after the
 * iterations.  Output in unit-variance units, ascending; distortion is
 * E‖u - û‖² for a unit vector u ([P1] Theorem 1 table).
 * Errors: INVALID_ARG for d < 2, b outside 1..4, NULL out, density unknown.
 */
typedef struct {
  int d, b, density, grid, iters;
  double centroid[16];  /* 2^b used */
  double threshold[15]; /* 2^b - 1 used, midpoints of consecutive centroids */
  double distortion;
} tq_codebook;

tq_status tq_codebook_build(int d, int b, int density, int grid, int iters, tq_codebook* out);

/* ------------------------------------------------------------------ rotation
 * Haar rotation from a Gaussian matrix: Π = Q · diag(sign(diag R)) for the
 * Householder QR G = Q R (sign(0) = +1).  [P1] section "TurboQuant_mse 的官方
 * 步骤" step 1 (QR of a Gaussian matrix); [P2] section "核心洞察" (generated
 * once from a fixed seed and shared by every vector).
 * h_G: d×d row-major fp64 (caller's seeded draw).  h_Pi: d×d row-major fp64
 * output.  Host only, synchronous.  Errors: INVALID_ARG (NULL, d < 1),
 * ALLOC (host memory).
 */
tq_status tq_rotation_haar(int d, const double* h_G, double* h_Pi);

/* ------------------------------------------------------------------ context
 * A context owns the device copies of everything a (d, b, mode, rotation)
 * needs: the rotation in the operand layouts of the kernels, the QJL matrix
 * (Prod), and the codebook tables.
 *
 * d, b      dimension and TOTAL bits per coordinate.  TQ_MSE quantizes with
 *           the b-bit codebook; TQ_PROD ([P1] section "TurboQuant_prod"; [P4]
 *           section "两阶段量化框架") uses a (b-1)-bit MSE stage plus 1 QJL bit.
 *           TQ_MIXED is TurboQuant_mse at b + 1/2 bits per coordinate ([P1]
 *           section "论文给出的关键数据点": 3.5 and 2.5 bit/channel; section
 *           "decode 阶段：写入少，但每步都要读取历史 cache": 672 B per token and
 *           layer = 16 vectors of 40 B of codes and a 2-byte norm): coordinate
 *           j of Π·u takes b + 1 bits where j mod 16 < 8 and b bits elsewhere,
 *           each half with the Lloyd-Max codebook of its own width (which half
 *           is immaterial: the coordinates of Π·u are exchangeable); b = 1..3
 *           (1.5, 2.5 or 3.5 bits), d = 128 (either rotation).
 * rot_kind  TQ_ROT_DENSE: h_rot is Π, d×d row-major fp64 (e.g. from
 *           tq_rotation_haar).  TQ_ROT_HADAMARD: h_rot is the sign vector σ
 *           (d entries ±1) and Π = H·diag(σ)/√d, H the Sylvester Hadamard
 *           matrix (d = 2^k) or H_12 ⊗ H_(d/12) (Paley q = 11 ⊗ Sylvester);
 *           [P3] chapters 3 and 7 (WHT rotation).
 * h_S       Prod only: the QJL matrix S, d×d row-major fp64 (i.i.d. N(0,1)),
 *           m = d rows.  NULL for TQ_MSE.
 * cb        codebook of the MSE stage: cb->d == d and cb->b == b (MSE) or
 *           b - 1 (Prod).  TQ_MIXED: an array of two codebooks, cb[0] with b
 *           bits and cb[1] with b + 1 bits, both for dimension d.  Copied; the
 *           caller may free it afterwards.
 * Synchronous.  Errors: INVALID_ARG, UNSUPPORTED (d or rot_kind), ALLOC, CUDA.
 */
typedef struct tq_ctx tq_ctx;

tq_status tq_ctx_create(int d, int b, int mode, int rot_kind, const double* h_rot,
                        const double* h_S, const tq_codebook* cb, tq_ctx** out);
tq_status tq_ctx_destroy(tq_ctx* ctx);

/* ------------------------------------------------------------------ codes
 * Packed codes of n vectors ([P1] section "一个具体例子" steps 4-6: indices
 * packed into a bit stream, the norm stored separately; [P3] chapter 3: read
 * as whole words, never byte by byte).
 *
 *   d_codes  uint32 words, words_per_vec per vector (16-byte multiple).
 *            TQ_LAYOUT_TOKEN: vector v's b_mse-bit code of coordinate j sits in
 *            bits [j*b_mse, (j+1)*b_mse) of its own stream, LSB first; stream
 *            bit p is bit p%32 of word p/32 (the canonical order).
 *            TQ_LAYOUT_PAIR: vectors 2i and 2i+1 share one block of
 *            2*words_per_vec words; coordinate j occupies bits
 *            [2*j*b_mse, 2*(j+1)*b_mse) of the block's stream, the even
 *            vector's code in the low b_mse bits.  (Used for V caches so that
 *            decode reads pairs of tokens per coordinate.)
 *            TQ_MIXED (b_mse = b): coordinate j's code has w_j bits (b + 1
 *            where j mod 16 < 8, else b) and occupies stream bits
 *            [P_j, P_j + w_j), P_j = w_0 + ... + w_(j-1); words_per_vec =
 *            d·(2b+1)/64 exactly (24, 40 or 56 bytes at d = 128, so vectors
 *            are 8-byte, not 16-byte, multiples).  PAIR: coordinate j holds a
 *            field of 2·w_j bits at block bit 2·P_j, the even vector's code
 *            in its low w_j bits.
 *   d_norm   fp32 ‖x‖ per vector.
 *   d_qjl    Prod only: d/32 words of sign bits per vector (bit j = [(S·r)_j >= 0]),
 *            padded to qjl_words_per_vec; NULL for MSE.
 *   d_rnorm  Prod only: fp32 residual norm γ = ‖r‖ per vector; NULL for MSE.
 *
 * tq_codes_layout fills every field except the four pointers and returns the
 * byte sizes to allocate for n vectors (PAIR: n rounded up to even).
 */
typedef struct {
  uint32_t* d_codes;
  float* d_norm;
  uint32_t* d_qjl;
  float* d_rnorm;
  int64_t n;
  int d, b_mse, mode, layout;
  int words_per_vec, qjl_words_per_vec;
} tq_codes;

tq_status tq_codes_layout(const tq_ctx* ctx, int layout, int64_t n, tq_codes* desc,
                          size_t* codes_bytes, size_t* norm_bytes, size_t* qjl_bytes,
                          size_t* rnorm_bytes);

/* ------------------------------------------------------------------ encode
 * Online TurboQuant encode of N vectors ([P1] section "一个具体例子" steps 1-6:
 * s = ‖x‖, u = x/s, y = Π·u, nearest codebook entry per coordinate, pack,
 * store s; [P1] section "TurboQuant_prod" for the residual r = u - Πᵀŷ,
 * γ = ‖r‖ and the 1-bit code sign(S·r) with sign(0) = +1).
 *
 * d_x       [N, d] row-major, fp32 (x_dtype TQ_F32) or fp16 (TQ_F16), 16-byte
 *           aligned.
 * out       destination codes (layout TOKEN or PAIR).  Row r of x is written
 *           to vector  (r / group_rows) * group_stride + offset + r % group_rows
 *           of out, which must be < out->n.  (group_rows = N, group_stride = 0
 *           writes rows contiguously from `offset`; group_rows = 1,
 *           group_stride = capacity appends one token to each (batch, head)
 *           block of a cache.)
 * A coordinate is coded as idx = #{k : v >= t_k}, i.e. the nearest centroid
 * with ties to the higher index.  A zero vector gets s = 0, all-zero codes,
 * γ = 0 and all-zero QJL bits.  In PAIR layout, writes of vectors whose
 * partner vector is not in the same call are read-modify-write with atomics;
 * calls that write the same pair block must be ordered on one stream.
 * d > 128 (MSE, TOKEN layout, d a multiple of 128 for the dense rotation;
 * TQ_ERR_UNSUPPORTED otherwise): two kernels on `stream`, a norm pass and a
 * tensor-core GEMM whose coordinates lying near a threshold are recomputed in
 * float-float arithmetic, so codes match the fp64 definition outside a band
 * of ~1e-6 around each threshold, as on every other path.  A context with the
 * randomized Hadamard rotation (MSE, d = 2^k or 12·2^k with 2^k in 32..256)
 * encodes with one kernel that applies the fast transform instead.
 * Norms: fp32 sums of squares; a vector whose sum leaves (1e-30, 1e36) is
 * summed again scaled by a power of two, so s is right for any finite
 * magnitude the input type can hold.
 */
tq_status tq_encode(const tq_ctx* ctx, const void* d_x, int x_dtype, int64_t N,
                    const tq_codes* out, int64_t offset, int64_t group_rows,
                    int64_t group_stride, tq_stream stream);

/* ------------------------------------------------------------------ scores
 * Inner-product scores of M queries against keys [first, first + N) of a code
 * set ([P4] section "工程实现的关键路径": pre-rotate the query once so each key
 * costs a table lookup and a dot product; [P1] and [P2] "内积偏差问题与 QJL
 * 修正器" for the Prod estimate).
 *   MSE :  score[m][n] = s_n · ⟨Π q_m, ŷ_n⟩
 *   Prod:  score[m][n] = s_n · (⟨Π q_m, ŷ_n⟩ + γ_n √(π/2)/d · ⟨S q_m, 2·bits_n − 1⟩)
 * d_q       [M, d] fp32 row-major.
 * keys      TOKEN layout.
 * d_scores  [M, N] fp32 row-major output.
 * d_ws      workspace of tq_scores_workspace_size bytes (16-byte aligned).
 */
tq_status tq_scores_workspace_size(const tq_ctx* ctx, int M, size_t* bytes);
tq_status tq_scores(const tq_ctx* ctx, const float* d_q, int M, const tq_codes* keys,
                    int64_t first, int64_t N, float* d_scores, void* d_ws, size_t ws_bytes,
                    tq_stream stream);

/* ------------------------------------------------------------------ decode
 * One decode step of attention over a TurboQuant_MSE KV cache
 * ([P1] section "decode 阶段到底怎么“用”这些压缩后的 KV", second route: unpack,
 * look up, scale and consume inside the attention kernel; [P3] chapter 1:
 * softmax(q Kᵀ / √d) V; [P4] section "工程实现的关键路径": pre-rotated query and
 * kv_head = q_head / (Hq / Hkv)).
 *   out[b][h] = Σ_t softmax_t(scale · ⟨q[b][h], k̂[b][kv][t]⟩) · v̂[b][kv][t],
 *   k̂ = s · Πᵀ ŷ, kv = h / (Hq / Hkv).
 * The value sum is accumulated in the rotated domain and rotated back once per
 * head at the end (linearity of Πᵀ).
 * Keys may be TurboQuant_Prod (kctx in TQ_PROD; [P1] section
 * "TurboQuant_prod", [P2] "内积偏差问题与 QJL 修正器"): then
 *   k̂ = s · (Πᵀ ŷ + γ · √(π/2)/d · Sᵀ (2·bits − 1)),
 * the unbiased inner-product estimate, computed as ⟨Π q, ŷ⟩ plus
 * γ·√(π/2)/d·⟨S q, 2·bits − 1⟩ with both query rotations done once per call.
 * K then needs its QJL words and γ (qjl, rnorm), and Hq / Hkv <= 4
 * (TQ_ERR_UNSUPPORTED otherwise).
 * kctx, vctx  contexts of the K (TQ_MSE, TQ_PROD or TQ_MIXED) and V (TQ_MSE
 *             or TQ_MIXED) codes; may be the same.  b + 1/2 bits ([P1]
 *             section "论文给出的关键数据点"): K and V both TQ_MIXED with the
 *             same b and codebooks, any GQA of 1, 2, 4, 8 (TQ_ERR_UNSUPPORTED
 *             otherwise).
 * d_q       [B, Hq, d], fp32 or fp16 (q_dtype).
 * K         TOKEN layout; V: PAIR layout.  Vector index of token t of
 *           (batch b, kv head h) is (b * Hkv + h) * cap + t; tokens [0, seq)
 *           are read.  cap must be even (TQ_ERR_INVALID_ARG) and a multiple
 *           of 16 (TQ_ERR_UNSUPPORTED otherwise).
 * d_out     [B, Hq, d] fp32.
 * d_ws      workspace of tq_decode_workspace_size bytes (16-byte aligned),
 *           zero-filled before its first use (e.g. cudaMemset).  It holds one
 *           arrival counter per (batch, KV head) and the partial softmax
 *           states of the CTAs that share a (batch, KV head); every call
 *           leaves the counters at zero again.  Calls that share a workspace
 *           must be ordered on one stream.
 * Hq % Hkv == 0 and Hq / Hkv in {1, 2, 4, 8}.
 */
tq_status tq_decode_workspace_size(const tq_ctx* kctx, int B, int Hq, int Hkv, int64_t seq,
                                   size_t* bytes);
tq_status tq_decode_attention(const tq_ctx* kctx, const tq_ctx* vctx, const void* d_q,
                              int q_dtype, const tq_codes* K, const tq_codes* V, int B, int Hq,
                              int Hkv, int64_t seq, int64_t cap, float scale, float* d_out,
                              void* d_ws, size_t ws_bytes, tq_stream stream);

/* ------------------------------------------------------------------ decode step
 * One decode step with the step's token appended first ([P1] section
 * "一个具体例子：KV Cache 在 prefill 和 decode 里怎么量化", decode: the token's K/V is
 * appended to the cache, then its query attends over the whole history).
 * d_k_new, d_v_new: [B, Hkv, d] (new_dtype fp32 or fp16, 16-byte aligned).
 * Encodes them as tq_encode does (norm, rotation, bucketize, pack; the same
 * codes except for coordinates within about 1e-6 of a codebook threshold,
 * where the two roundings may fall on either side, and the same norm to fp32
 * rounding) into position seq-1 of every (batch, KV head) block of K and V,
 * then computes tq_decode_attention over tokens [0, seq) including the new
 * one, in one kernel launch.  Keys must be TurboQuant_MSE here
 * (TQ_ERR_UNSUPPORTED for TQ_PROD and TQ_MIXED: append with tq_encode, then call
 * tq_decode_attention).  Other arguments, the workspace and errors as
 * tq_decode_attention.  The V pair block of position seq-1 is updated with atomics, so
 * its partner token (seq-2 or seq) may be written by an ordered earlier call.
 */
tq_status tq_decode_step(const tq_ctx* kctx, const tq_ctx* vctx, const void* d_q, int q_dtype,
                         const void* d_k_new, const void* d_v_new, int new_dtype, const tq_codes* K,
                         const tq_codes* V, int B, int Hq, int Hkv, int64_t seq, int64_t cap,
                         float scale, float* d_out, void* d_ws, size_t ws_bytes,
                         tq_stream stream);

/* ------------------------------------------------------------------ decode, no workspace
 * The pages have no counterpart to this call; it exists for callers that
 * cannot allocate device memory: code running where cudaMalloc is unavailable
 * or forbidden (inside a host callback or a driver-managed region, a fixed
 * memory-budget runtime, or a plugin that may not own allocations) and so
 * cannot hand tq_decode_attention a workspace either.
 *
 * Same computation, arguments and results as tq_decode_attention, minus d_ws
 * and ws_bytes.  Its scratch (the counters and partial softmax states that
 * tq_decode_attention keeps in the workspace) is a 2 MiB array built into the
 * library, which every GPU that loads libtq keeps reserved until the process
 * exits.
 *   - Shapes whose scratch (tq_decode_workspace_size) exceeds 2 MiB return
 *     TQ_ERR_UNSUPPORTED before anything is launched.  The need is 4 bytes per
 *     (batch, KV head) plus at most about 80 KB per query head of a KV head
 *     (0.3 MB for 8 KV heads with 4 query heads each, at any sequence length).
 *   - The first call on a device looks up the array's device address (once per
 *     device, with that device current); make that first call before any stream
 *     capture.
 *   - All calls share the array: two calls that overlap on the GPU (different
 *     streams, no ordering between them) race and corrupt each other's output.
 *     Order them on one stream.  Each call first zeroes the array's arrival
 *     counters on `stream` (a memset, which allocates nothing), so a call that
 *     failed part-way leaves nothing behind for the next one; every other
 *     state a call reads it writes itself first.
 * The call itself allocates nothing (no cudaMalloc or allocating library routine).
 */
tq_status tq_decode_attention_noalloc(const tq_ctx* kctx, const tq_ctx* vctx, const void* d_q,
                                      int q_dtype, const tq_codes* K, const tq_codes* V, int B,
                                      int Hq, int Hkv, int64_t seq, int64_t cap, float scale,
                                      float* d_out, tq_stream stream);

/* ------------------------------------------------------------------ views
 * Canonical view of stored codes, for checking: copies vectors
 * [first, first + count) to the host and writes their coordinate indices
 * (h_idx, count × d bytes) and, for Prod, their QJL bits (h_bits, count × d
 * bytes of 0/1; may be NULL).  Synchronous (device-wide copy).
 */
tq_status tq_unpack_indices(const tq_codes* codes, int64_t first, int64_t count, uint8_t* h_idx,
                            uint8_t* h_bits);

/* Bound of the pipeline waits (mbarrier phases) of the tensor-memory kernels
 * launched with this context afterwards (the encoders for d = 128 and
 * d > 128 with the dense rotation, and the scorer): a wait that has polled `polls` times without success gives up; the
 * kernel then stops its pipeline, waits (with the default bound) for its own
 * copies and tensor-core operations in flight, frees its tensor memory and
 * returns, leaving its outputs unspecified, and tq_status_poll reports
 * TQ_ERR_TIMEOUT once.  Default 2^22 polls (seconds); 0 makes every such wait
 * give up before its first poll, which exercises that path on demand.  A
 * failure-handling and testing aid: not synchronised with launches in flight,
 * so set it between calls.  Errors: INVALID_ARG (NULL ctx). */
tq_status tq_ctx_set_wait_limit(tq_ctx* ctx, uint32_t polls);

/* Reads and clears the context's device status word (synchronises `stream`).
 * Returns TQ_OK, or TQ_ERR_TIMEOUT if a bounded device wait of a kernel
 * launched with this context ran out since the last poll (that kernel's
 * outputs are then unspecified). */
tq_status tq_status_poll(const tq_ctx* ctx, tq_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* TQ_H_ */
