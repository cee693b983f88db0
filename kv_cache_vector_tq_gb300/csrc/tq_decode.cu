// Host side of decode attention: parameters, the launch, and the variant
// without a workspace.  The kernel is in tq_decode_kernel.cuh.
#include <mutex>

#include "tq_decode_kernel.cuh"

namespace tq {

size_t decode_ws_bytes(int d, int B, int Hq, int Hkv, int64_t seq) {
  (void)d;
  (void)seq;
  if (B <= 0 || Hq <= 0 || Hkv <= 0) return 256;
  const int G = Hq / Hkv;
  return ws_counter_bytes(B * Hkv) + (size_t)num_sms() * G * kPart * sizeof(float) + 256;
}


tq_status launch_step(const DevCtx& kc, const DevCtx& vc, const void* q, int q_dtype,
                      const void* knew, const void* vnew, int new_dtype, const tq_codes* K,
                      const tq_codes* V, int B, int Hq, int Hkv, int64_t seq, int64_t cap,
                      float scale, float* out, void* ws, cudaStream_t stream) {
  if (cap % 16 != 0) return TQ_ERR_UNSUPPORTED;
  // b + 1/2 bits: K and V both, equal b and identical tables, in the attention
  // entry (append with tq_encode first)
  const bool mixed = kc.mode == TQ_MIXED || vc.mode == TQ_MIXED;
  if (mixed) {
    bool same = kc.mode == vc.mode && kc.b_mse == vc.b_mse && kc.alpha == vc.alpha && knew == nullptr;
    for (int k = 0; same && k < (1 << kc.b_mse); ++k) same = kc.cen[k] == vc.cen[k];
    for (int k = 0; same && k < (2 << kc.b_mse); ++k) same = kc.cen_hi[k] == vc.cen_hi[k];
    if (!same) return TQ_ERR_UNSUPPORTED;
  }
  const int G = Hq / Hkv;
  const bool prod = kc.mode == TQ_PROD;
  if (prod && (knew != nullptr || G > 4 || kc.b_mse > 3 || !kc.s_slices || !K->d_qjl || !K->d_rnorm ||
               K->qjl_words_per_vec != 4))
    return TQ_ERR_UNSUPPORTED;
  bool same_lut = kc.b_mse == vc.b_mse && kc.alpha == vc.alpha;
  for (int k = 0; same_lut && k < (1 << kc.b_mse); ++k) same_lut = kc.cen[k] == vc.cen[k];
  StepParams p;
  p.kslices = kc.pi_slices;
  p.vslices = vc.pi_slices;
  p.vpi = vc.pi;
  p.status = kc.status;
  p.klut = kc.lut;
  p.vlut = vc.lut;
  p.klut_hi = kc.lut_hi;
  p.same_lut = same_lut ? 1 : 0;
  for (int k = 0; k < 15; ++k) {
    p.kthr[k] = kc.thr[k];
    p.vthr[k] = vc.thr[k];
  }
  p.kfold = scale * kLog2e / (kc.sqrt_d * kc.alpha);
  p.qfold = prod ? (float)(scale * kLog2e * std::sqrt(3.14159265358979323846 / 2.0) / kc.d) : 0.f;
  p.sslices = prod ? kc.s_slices : nullptr;
  p.kqjl = prod ? K->d_qjl : nullptr;
  p.krn = prod ? K->d_rnorm : nullptr;
  p.vfold = 1.f / (vc.alpha * vc.sqrt_d);
  p.sqrt_d = kc.sqrt_d;
  p.kcodes = K->d_codes;
  p.knorm = K->d_norm;
  p.vcodes = V->d_codes;
  p.vnorm = V->d_norm;
  p.seq = seq;
  p.cap = cap;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.tiles = (int)((seq + kTileTok - 1) / kTileTok);
  p.q = q;
  p.q_f16 = q_dtype == TQ_F16;
  p.knew = knew;
  p.vnew = vnew;
  p.new_f16 = new_dtype == TQ_F16;
  p.append = knew != nullptr;
  p.out = out;
  int groups = B * Hkv;
  p.kv_shift = 0;
  // 8 query heads per KV head over short caches: as 4-head groups over two
  // virtual KV heads per cache head (the 8-head kernel needs ~230 registers and
  // so runs 8 warps per SM; the 4-head one runs 16).  Both halves read the same
  // cache bytes, the second mostly from L2 while the cache is short: 64 q / 8
  // kv heads at b = 3, 4096 tokens 12.6 -> 9.8 us, but 16384 tokens 18.5 ->
  // 20.5 us and 131072 tokens 65.7 -> 100 us (the second reads miss L2).
  int Gk = G;
  if (G == 8 && !prod && !mixed && 2 * groups <= num_sms() && seq <= 4096) {
    Gk = 4;
    groups *= 2;
    p.Hkv = 2 * Hkv;
    p.kv_shift = 1;
  }
  p.S = 1;
  p.counters = static_cast<int*>(ws);
  p.part = reinterpret_cast<float*>(static_cast<char*>(ws) + ws_counter_bytes(groups));
  cudaError_t e;
  if (mixed)
    e = decode_run_mixed(p, kc.b_mse, G, groups, stream);
  else if (prod)
    e = decode_run_prod(p, kc.b_mse, vc.b_mse, G, groups, stream);
  else if (kc.b_mse == 1)
    e = decode_run_k1(p, vc.b_mse, Gk, groups, stream);
  else if (kc.b_mse == 2)
    e = decode_run_k2(p, vc.b_mse, Gk, groups, stream);
  else if (kc.b_mse == 3)
    e = decode_run_k3(p, vc.b_mse, Gk, groups, stream);
  else if (kc.b_mse == 4)
    e = decode_run_k4(p, vc.b_mse, Gk, groups, stream);
  else
    return TQ_ERR_UNSUPPORTED;
  return e == cudaSuccess ? TQ_OK : set_cuda_error(e);
}

tq_status launch_decode(const DevCtx& kc, const DevCtx& vc, const void* q, int q_dtype,
                        const tq_codes* K, const tq_codes* V, int B, int Hq, int Hkv, int64_t seq,
                        int64_t cap, float scale, float* out, void* ws, size_t ws_bytes,
                        cudaStream_t stream) {
  (void)ws_bytes;
  return launch_step(kc, vc, q, q_dtype, nullptr, nullptr, TQ_F16, K, V, B, Hq, Hkv, seq, cap,
                     scale, out, ws, stream);
}

// ------------------------------------------------------------------ decode without a workspace
// Scratch for tq_decode_attention_noalloc: the arrival counters and partial
// softmax states that tq_decode_attention keeps in the caller's workspace.  It
// is a file-scope device array, so the driver reserves it on every GPU that
// loads the library, and it stays reserved until the process exits.  It starts
// zero-filled and every call leaves the counters at zero; concurrent calls (on
// different streams) would race on it.
constexpr size_t kNoAllocScratchBytes = (size_t)2 << 20;  // 2 MiB
static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

size_t decode_noalloc_limit() { return kNoAllocScratchBytes; }

// Device address of the scratch array on the current device.  The host-side
// symbol is only a stand-in, so the address is asked from the runtime once per
// device (with that device current) and cached.
static cudaError_t decode_scratch_address(void** out) {
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
  // Every call that completes leaves the counters at zero, but a call that
  // failed part-way could leave them set, and the caller cannot reach this
  // array to clear it: zero them on the call's stream first (no allocation).
  e = cudaMemsetAsync(ws, 0, ws_counter_bytes(B * Hkv), stream);
  if (e != cudaSuccess) return set_cuda_error(e);
  return launch_decode(kc, vc, q, q_dtype, K, V, B, Hq, Hkv, seq, cap, scale, out, ws, need, stream);
}

}  // namespace tq