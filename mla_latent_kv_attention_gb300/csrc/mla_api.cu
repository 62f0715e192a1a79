// mla_api.cu -- the C ABI of libmla: argument checks, workspace layout, launches.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "mla_internal.cuh"

namespace {

thread_local int g_last_launches = 0;
thread_local cudaEvent_t g_prof_start = nullptr, g_prof_stop = nullptr;
thread_local unsigned long long* g_trace = nullptr;  // mla_set_trace_buffer
thread_local int g_trace_ctas = 0;

void prof_mark(cudaEvent_t e, cudaStream_t s) {
  if (g_prof_start && g_prof_stop) cudaEventRecord(e, s);
}

int sm_count(int device) {
  static int cache[64] = {0};
  if (device >= 0 && device < 64 && cache[device] > 0) return cache[device];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  if (device >= 0 && device < 64) cache[device] = n;
  return n;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

mla_status_t check_kv(const mla_kv_t* kv) {
  if (!kv || !kv->pool || !kv->page_table || !kv->seq_lens) return MLA_ERR_INVALID_ARG;
  if (kv->num_pages < 0 || kv->page_table_stride < 1) return MLA_ERR_INVALID_ARG;
  if (kv->page_size <= 0 || kv->page_size % 64 != 0) return MLA_ERR_UNSUPPORTED;
  if (!aligned(kv->pool, 16) || !aligned(kv->page_table, 4) || !aligned(kv->seq_lens, 4))
    return MLA_ERR_INVALID_ARG;
  return MLA_OK;
}

mla::AttnParams base_params(const mla_kv_t* kv, const void* q, int B, int n_q, int H,
                            float sm_scale, void* out, float* lse) {
  mla::AttnParams p = {};
  p.pool = kv->pool;
  p.num_pages = kv->num_pages;
  p.page_size = kv->page_size;
  p.page_table = kv->page_table;
  p.pt_stride = kv->page_table_stride;
  p.seq_lens = kv->seq_lens;
  p.kv_scale = kv->kv_scale;
  p.sm_scale = sm_scale;
  p.q = static_cast<const uint16_t*>(q);
  p.B = B;
  p.n_q = n_q;
  p.H = H;
  p.R = n_q * H;
  p.part_rows = p.R;
  p.out = static_cast<uint16_t*>(out);
  p.lse = lse;
  p.trace = g_trace;
  p.trace_ctas = g_trace_ctas;
  return p;
}

mla_status_t current_device(int* dev) {
  if (cudaGetDevice(dev) != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  return MLA_OK;
}

// Set by mla_test_stall_next_call; consumed (and cleared) by the next decode/verify call on
// this thread.
thread_local int g_test_stall = 0;

mla_status_t run_split(const mla_kv_t* kv, const void* q, int B, int n_q, int H, float sm_scale,
                       void* out, float* lse, void* ws, size_t ws_bytes, void* stream,
                       bool out_is_f32 = false, int mask_shift = 0) {
  g_last_launches = 0;
  mla_status_t st = check_kv(kv);
  if (st != MLA_OK) return st;
  if (B < 0) return MLA_ERR_INVALID_ARG;
  if (H < 1 || H > MLA_MAX_HEADS || n_q < 1 || n_q > MLA_MAX_NQ) return MLA_ERR_UNSUPPORTED;
  if (!q || !out) return MLA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(out, 16) || (lse && !aligned(lse, 4))) return MLA_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, 256)) return MLA_ERR_WORKSPACE;
  int dev;
  if ((st = current_device(&dev)) != MLA_OK) return st;
  const int sms = sm_count(dev);
  if (sms <= 0) return MLA_ERR_CUDA;
  const mla::WsLayout w = mla::ws_layout(B, n_q * H, sms);
  if (ws_bytes < w.total) return MLA_ERR_WORKSPACE;
  if (B == 0) return MLA_OK;
  mla::AttnParams p = base_params(kv, q, B, n_q, H, sm_scale, out, lse);
  p.test_stall = g_test_stall;
  g_test_stall = 0;
  p.mask_shift = mask_shift;
  if (out_is_f32) {
    p.out = nullptr;
    p.out_f32 = static_cast<float*>(out);
  }
  char* base = static_cast<char*>(ws);
  p.hdr = reinterpret_cast<mla::WsHeader*>(base + w.hdr);
  p.status = reinterpret_cast<unsigned*>(base + w.status);
  p.part_lse = reinterpret_cast<float*>(base + w.part_lse);
  p.part_out = reinterpret_cast<float*>(base + w.part_out);
  p.qimg = reinterpret_cast<uint8_t*>(base + w.qimg);
  p.qimg_stride = (int64_t)w.qimg_stride;
  p.num_ctas = sms;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  prof_mark(g_prof_start, s);
  int launched = 0;
  const cudaError_t e = mla::launch_decode_tc(p, sms, s, &launched);
  g_last_launches += launched;
  if (e != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  prof_mark(g_prof_stop, s);
  if (mla::launch_merge(p, s) != cudaSuccess) return MLA_ERR_CUDA;
  ++g_last_launches;
  return MLA_OK;
}

}  // namespace

extern "C" {

size_t mla_workspace_size(mla_op_t op, int B, int H, int n_q, int device) {
  if (H < 1 || H > MLA_MAX_HEADS || B < 0) return 0;
  if (op == MLA_OP_PREFILL) {
    if (B != 1 || n_q < 0) return 0;
    const int sms = sm_count(device);
    return sms > 0 ? mla::ws_prefill_bytes(sms) : 0;
  }
  if (op == MLA_OP_DECODE) n_q = 1;
  if (n_q < 1 || n_q > MLA_MAX_NQ) return 0;
  const int sms = sm_count(device);
  if (sms <= 0) return 0;
  return mla::ws_layout(B, n_q * H, sms).total;
}

mla_status_t mla_decode(const mla_kv_t* kv, const void* q, int B, int H, float sm_scale,
                        void* out, float* lse, void* workspace, size_t workspace_bytes,
                        void* stream) {
  return run_split(kv, q, B, 1, H, sm_scale, out, lse, workspace, workspace_bytes, stream);
}

mla_status_t mla_verify(const mla_kv_t* kv, const void* q, int B, int n_q, int H,
                        float sm_scale, void* out, float* lse, void* workspace,
                        size_t workspace_bytes, void* stream) {
  return run_split(kv, q, B, n_q, H, sm_scale, out, lse, workspace, workspace_bytes, stream);
}

mla_status_t mla_verify_f32(const mla_kv_t* kv, const void* q, int B, int n_q, int H,
                            float sm_scale, float* out, float* lse, void* workspace,
                            size_t workspace_bytes, void* stream) {
  return run_split(kv, q, B, n_q, H, sm_scale, out, lse, workspace, workspace_bytes, stream, true);
}

mla_status_t mla_verify_f32_shard(const mla_kv_t* kv, const void* q, int B, int n_q, int H,
                                  float sm_scale, int visible_shift, float* out, float* lse,
                                  void* workspace, size_t workspace_bytes, void* stream) {
  if (visible_shift < 0) return MLA_ERR_INVALID_ARG;
  const int shift = (n_q >= 1 && visible_shift > n_q - 1) ? n_q - 1 : visible_shift;
  return run_split(kv, q, B, n_q, H, sm_scale, out, lse, workspace, workspace_bytes, stream, true,
                   shift);
}

size_t mla_prefill_mha_workspace_size(int L, int H, int device) {
  if (L < 0 || H < 1 || H > MLA_MAX_HEADS) return 0;
  const int sms = sm_count(device);
  if (sms <= 0) return 0;
  return mla::mha_ws_layout(L, H, sms).total;
}

namespace {

mla_status_t run_mha(const mla_kv_t* kv, int L, const void* q, int T, int H, const void* w_ukv,
                     float sm_scale, void* out, float* lse, void* workspace,
                     size_t workspace_bytes, void* stream, int precise) {
  g_last_launches = 0;
  mla_status_t st = check_kv(kv);
  if (st != MLA_OK) return st;
  if (T < 0 || L < T) return MLA_ERR_INVALID_ARG;
  if (H < 1 || H > MLA_MAX_HEADS) return MLA_ERR_UNSUPPORTED;
  if (!q || !w_ukv || !out) return MLA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(w_ukv, 16) || !aligned(out, 16) || (lse && !aligned(lse, 4)))
    return MLA_ERR_INVALID_ARG;
  if ((int64_t)L > kv->page_table_stride * (int64_t)kv->page_size) return MLA_ERR_INVALID_ARG;
  if (!workspace || !aligned(workspace, 256)) return MLA_ERR_WORKSPACE;
  if (workspace_bytes < sizeof(mla::WsHeader)) return MLA_ERR_WORKSPACE;
  if (T == 0) return MLA_OK;
  int dev;
  if ((st = current_device(&dev)) != MLA_OK) return st;
  const int sms = sm_count(dev);
  if (sms <= 0) return MLA_ERR_CUDA;
  const mla::MhaWsLayout w = mla::mha_ws_layout(L, H, sms);
  if (workspace_bytes < w.total) return MLA_ERR_WORKSPACE;
  char* base = static_cast<char*>(workspace);
  mla::MhaArgs a;
  a.pool = kv->pool;
  a.num_pages = kv->num_pages;
  a.page_size = kv->page_size;
  a.page_table = kv->page_table;
  a.kv_scale = kv->kv_scale;
  a.L = L;
  a.T = T;
  a.H = H;
  a.sm_scale = sm_scale;
  a.q = q;
  a.w_ukv = w_ukv;
  a.latent = base + w.latent;
  a.rope = base + w.rope;
  a.kvup = base + w.kvup;
  a.part_out = base + w.part_out;
  a.part_lse = base + w.part_lse;
  a.out = static_cast<uint16_t*>(out);
  a.lse = lse;
  a.status = reinterpret_cast<unsigned*>(base + w.status);
  a.hdr = reinterpret_cast<mla::WsHeader*>(base);
  a.device = dev;
  a.precise = precise;
  a.prof_start = g_prof_start;  // the profiling events bracket the attention kernel alone
  a.prof_stop = g_prof_stop;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int launched = 0;
  const cudaError_t e = mla::launch_mha_prefill(a, sms, s, &launched);
  g_last_launches += launched;
  if (e != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  return MLA_OK;
}

}  // namespace

mla_status_t mla_prefill_mha(const mla_kv_t* kv, int L, const void* q, int T, int H,
                             const void* w_ukv, float sm_scale, void* out, float* lse,
                             void* workspace, size_t workspace_bytes, void* stream) {
  return run_mha(kv, L, q, T, H, w_ukv, sm_scale, out, lse, workspace, workspace_bytes, stream, 1);
}

mla_status_t mla_prefill_mha_bf16(const mla_kv_t* kv, int L, const void* q, int T, int H,
                                  const void* w_ukv, float sm_scale, void* out, float* lse,
                                  void* workspace, size_t workspace_bytes, void* stream) {
  return run_mha(kv, L, q, T, H, w_ukv, sm_scale, out, lse, workspace, workspace_bytes, stream, 0);
}

mla_status_t mla_prefill(const mla_kv_t* kv, const void* q, int T, int H, float sm_scale,
                         void* out, float* lse, void* workspace, size_t workspace_bytes,
                         void* stream) {
  g_last_launches = 0;
  mla_status_t st = check_kv(kv);
  if (st != MLA_OK) return st;
  if (T < 0) return MLA_ERR_INVALID_ARG;
  if (H < 1 || H > MLA_MAX_HEADS) return MLA_ERR_UNSUPPORTED;
  if (!q || !out) return MLA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(out, 16) || (lse && !aligned(lse, 4))) return MLA_ERR_INVALID_ARG;
  if (!workspace || !aligned(workspace, 256)) return MLA_ERR_WORKSPACE;
  if (workspace_bytes < sizeof(mla::WsHeader)) return MLA_ERR_WORKSPACE;
  if (T == 0) return MLA_OK;
  int dev;
  if ((st = current_device(&dev)) != MLA_OK) return st;
  const int sms = sm_count(dev);
  if (sms <= 0) return MLA_ERR_CUDA;
  if (workspace_bytes < mla::ws_prefill_bytes(sms)) return MLA_ERR_WORKSPACE;
  mla::AttnParams p = base_params(kv, q, 1, T, H, sm_scale, out, lse);
  char* base = static_cast<char*>(workspace);
  p.hdr = reinterpret_cast<mla::WsHeader*>(base);
  p.status = reinterpret_cast<unsigned*>(base + mla::ws_prefill_status(sms));
  p.qimg = reinterpret_cast<uint8_t*>(base + mla::ws_prefill_qimg(sms));
  p.qimg_stride = (int64_t)mla::qimg_bytes(48);
  p.part_lse = reinterpret_cast<float*>(base + mla::ws_prefill_part_lse(sms));
  p.part_out = reinterpret_cast<float*>(base + mla::ws_prefill_part_out(sms));
  p.part_rows = 48;
  p.num_ctas = sms;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  prof_mark(g_prof_start, s);
  int launched = 0;
  const cudaError_t e = mla::launch_prefill_tc(p, sms, s, &launched);
  g_last_launches += launched;
  if (e != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  prof_mark(g_prof_stop, s);
  return MLA_OK;
}

mla_status_t mla_merge_lse(const float* part_out, const float* part_lse, int S, int64_t R,
                           void* out, float* lse, void* stream) {
  g_last_launches = 0;
  if (S < 0 || R < 0) return MLA_ERR_INVALID_ARG;
  if (R == 0) return MLA_OK;
  if (!out || (S > 0 && (!part_out || !part_lse))) return MLA_ERR_INVALID_ARG;
  if (!aligned(part_out, 16) || !aligned(part_lse, 4) || !aligned(out, 8) ||
      (lse && !aligned(lse, 4)))
    return MLA_ERR_INVALID_ARG;
  if (R > 0x7fffffff) return MLA_ERR_UNSUPPORTED;
  int dev;
  mla_status_t st = current_device(&dev);
  if (st != MLA_OK) return st;
  const int sms = sm_count(dev);
  if (sms <= 0) return MLA_ERR_CUDA;
  if (mla::launch_merge_standalone(part_out, part_lse, S, R, static_cast<uint16_t*>(out), lse, sms,
                                   static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MLA_ERR_CUDA;
  ++g_last_launches;
  return MLA_OK;
}

mla_status_t mla_cache_append(uint8_t* pool, int64_t num_pages, int32_t page_size,
                              const void* x, const int64_t* slots, int64_t n, float kv_scale,
                              unsigned* status, void* stream) {
  g_last_launches = 0;
  if (n < 0 || num_pages < 0 || page_size <= 0) return MLA_ERR_INVALID_ARG;
  if (!(kv_scale > 0.f) || !(kv_scale < INFINITY)) return MLA_ERR_INVALID_ARG;
  if (n == 0) return MLA_OK;
  if (!pool || !x || !slots) return MLA_ERR_INVALID_ARG;
  if (!aligned(pool, 16) || !aligned(x, 16) || !aligned(slots, 8) || (status && !aligned(status, 4)))
    return MLA_ERR_INVALID_ARG;
  int dev;
  mla_status_t st = current_device(&dev);
  if (st != MLA_OK) return st;
  const int sms = sm_count(dev);
  if (sms <= 0) return MLA_ERR_CUDA;
  const float inv = 1.0f / kv_scale;  // binary32, as the definition states
  if (mla::launch_cache_append(pool, num_pages * (int64_t)page_size, static_cast<const uint16_t*>(x),
                               slots, n, inv, status, sms, static_cast<cudaStream_t>(stream)) !=
      cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  ++g_last_launches;
  return MLA_OK;
}

mla_status_t mla_top_k_renorm_prob(const float* probs, float* out, int B, int V,
                                   const int32_t* top_k, int k, void* stream) {
  g_last_launches = 0;
  if (B < 0 || V < 0) return MLA_ERR_INVALID_ARG;
  if (B == 0 || V == 0) return MLA_OK;
  if (!probs || !out || !aligned(probs, 4) || !aligned(out, 4) || (top_k && !aligned(top_k, 4)))
    return MLA_ERR_INVALID_ARG;
  if (mla::launch_top_k_renorm(probs, out, B, V, top_k, k, static_cast<cudaStream_t>(stream)) !=
      cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  ++g_last_launches;
  return MLA_OK;
}

void mla_test_stall_next_call(void) { g_test_stall = 1; }

mla_status_t mla_read_status(const void* workspace, size_t workspace_bytes, void* stream) {
  if (!workspace || workspace_bytes < sizeof(mla::WsHeader)) return MLA_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  mla::WsHeader h;
  if (cudaMemcpyAsync(&h, workspace, sizeof(h), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  // one word per CTA of the last launch, right after the header; the first error wins
  const size_t off = mla::align_up(sizeof(mla::WsHeader), 256);
  if (h.num_ctas < 0 || h.num_ctas > 4096 || off + sizeof(unsigned) * (size_t)h.num_ctas > workspace_bytes)
    return MLA_ERR_WORKSPACE;
  if (h.num_ctas == 0) return MLA_OK;
  unsigned words[4096];
  if (cudaMemcpyAsync(words, static_cast<const char*>(workspace) + off,
                      sizeof(unsigned) * (size_t)h.num_ctas, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  for (int c = 0; c < h.num_ctas; ++c)
    if (words[c] != 0) return static_cast<mla_status_t>(words[c]);
  return MLA_OK;
}

const char* mla_status_string(mla_status_t status) {
  switch (status) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG: null, negative or misaligned argument";
    case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED: heads, positions or page size out of range";
    case MLA_ERR_WORKSPACE: return "MLA_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case MLA_ERR_CUDA: return "MLA_ERR_CUDA: a CUDA runtime call failed";
    case MLA_ERR_TIMEOUT: return "MLA_ERR_TIMEOUT: a bounded wait inside a kernel gave up";
    case MLA_ERR_BOUNDS: return "MLA_ERR_BOUNDS: page index outside the pool or length beyond the page table";
  }
  return "unknown mla_status_t";
}

int mla_last_launch_count(void) { return g_last_launches; }

void mla_set_profile_events(void* start, void* stop) {
  g_prof_start = static_cast<cudaEvent_t>(start);
  g_prof_stop = static_cast<cudaEvent_t>(stop);
}

void mla_set_trace_buffer(void* device_buffer, size_t bytes) {
  const size_t per_cta = sizeof(unsigned long long) * mla::kTraceWords;
  g_trace = (device_buffer && bytes >= per_cta) ? static_cast<unsigned long long*>(device_buffer) : nullptr;
  g_trace_ctas = g_trace ? (int)(bytes / per_cta < 65536 ? bytes / per_cta : 65536) : 0;
}

}  // extern "C"
