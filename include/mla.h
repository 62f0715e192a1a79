/*
 * mla.h -- C ABI of libmla: Multi-head Latent Attention (MLA) over a paged FP8-e4m3
 * latent KV cache, for one GB300 (sm_103a) GPU.
 *
 * The operation (all entry points): every cached position is one row of 576 e4m3 codes,
 * read as a 512-wide latent followed by a 64-wide RoPE part. Keys are whole rows, values
 * their first 512 entries, both dequantised as e4m3(code) * kv_scale ("MI355X Kimi K2.5
 * vLLM AITER 7x speedup", section "PR #35850 修复了什么": keys and values share one latent
 * space, FP8 KV cache; "Scaling Kimi K3 on AMD Instinct MI355X", section
 * "缓存可复用，还要能一致地恢复": 576 FP8 bytes per position). For query row
 * (sequence b, new position j, head h) with bfloat16 query q[576]:
 *     s_n   = sm_scale * sum_d q[d] * k_n[d]                 for visible keys n
 *     lse   = ln sum_n exp(s_n)                              (natural log, float32)
 *     out   = sum_n exp(s_n - lse) * v_n                     (bfloat16, round to nearest even)
 * Key n is visible to new position j iff n <= seq_lens[b] - n_q + j: the n_q new positions
 * are already written to the cache and are causal among themselves. Heads attend
 * independently ("Scaling Kimi K3 ...", section "并行度必须适配真正的形状"), so any
 * head count 1..16 runs as is; nothing is padded in memory.
 *
 * Conventions for every entry point:
 *  - Pointers marked "device" point to GPU global memory the caller owns; the library
 *    never allocates, frees or synchronises on the compute entry points. All work is
 *    enqueued on `stream` (a cudaStream_t passed as void*; NULL = legacy default stream)
 *    and is stream-ordered with the caller's other work.
 *  - bfloat16 tensors are passed as their 16-bit patterns (uint16_t / void*).
 *  - Argument errors the host can see return an error status immediately and enqueue
 *    nothing. Errors only the GPU can see (a page index outside the pool, a length larger
 *    than the page table holds, a bounded wait that gave up) are written to a status word
 *    inside the workspace and read back with mla_read_status(). No entry point aborts,
 *    asserts or traps.
 *  - Layouts are dense, row-major, with the innermost dimension last as written.
 */
#ifndef MLA_H
#define MLA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MLA_D 576       /* e4m3 codes per cached position (512 latent + 64 RoPE) */
#define MLA_DV 512      /* value width: the first 512 codes of a row              */
#define MLA_MAX_HEADS 16
#define MLA_MAX_NQ 4    /* verify positions per sequence                          */

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1, /* null pointer, negative size, misaligned pointer          */
  MLA_ERR_UNSUPPORTED = 2, /* heads outside 1..16, n_q outside 1..4, page size not 64k */
  MLA_ERR_WORKSPACE = 3,   /* workspace missing or smaller than mla_workspace_size()   */
  MLA_ERR_CUDA = 4,        /* a CUDA runtime call failed (launch, attribute query)      */
  MLA_ERR_TIMEOUT = 5,     /* device: a bounded wait inside a kernel gave up           */
  MLA_ERR_BOUNDS = 6       /* device: page index outside the pool or length > table    */
} mla_status_t;

typedef enum { MLA_OP_DECODE = 0, MLA_OP_VERIFY = 1, MLA_OP_PREFILL = 2 } mla_op_t;

/*
 * The paged latent cache.
 *   pool              device, [num_pages][page_size][576] e4m3 codes; 16-byte aligned.
 *   num_pages         pages in the pool (page indices must lie in [0, num_pages)).
 *   page_size         positions per page; 64 or a multiple of 64.
 *   page_table        device, [B][page_table_stride] int32: physical page of logical page p
 *                     of sequence b. Entries past a sequence's last page are never read.
 *   page_table_stride entries per row of page_table (>= pages of the longest sequence).
 *   seq_lens          device, [B] int32: cached positions of each sequence, including the
 *                     n_q new ones. 0 is allowed (the rows come out as out = 0,
 *                     lse = -inf). Negative or larger than page_table_stride * page_size:
 *                     MLA_ERR_BOUNDS in the status word, that sequence treated as empty.
 *   kv_scale          dequantised value = e4m3(code) * kv_scale, for K and V alike.
 * A contiguous cache is the identity page table.
 */
typedef struct mla_kv {
  const uint8_t* pool;
  int64_t num_pages;
  int32_t page_size;
  const int32_t* page_table;
  int64_t page_table_stride;
  const int32_t* seq_lens;
  float kv_scale;
} mla_kv_t;

/*
 * Bytes of workspace the given call needs on `device` (a CUDA ordinal). The workspace
 * holds the per-split partial outputs, staged query rows and one status word per CTA (it
 * depends on H, n_q and the SM count, not on B); it must be 256-byte aligned and stay untouched until the call's
 * work has finished on its stream. Its contents need no initialisation: every call
 * rewrites all it later reads (zero-fill it once if mla_read_status may run before the
 * first call). For MLA_OP_PREFILL pass B = 1 and n_q = T. Returns 0 for unsupported
 * arguments.
 */
size_t mla_workspace_size(mla_op_t op, int B, int H, int n_q, int device);

/*
 * Decode: one new position per sequence (n_q = 1).
 *   q    device, [B][H][576] bfloat16, 16-byte aligned
 *   out  device, [B][H][512] bfloat16
 *   lse  device, [B][H] float32 (natural log); may be NULL if not wanted
 * The key axis of long sequences is split across the GPU's SMs; per-split results are
 * combined with the log-sum-exp merge ("Scaling Kimi K3 ...", section
 * "缓存可复用，还要能一致地恢复": partial attention merged by normalisation statistics).
 */
mla_status_t mla_decode(const mla_kv_t* kv, const void* q, int B, int H, float sm_scale,
                        void* out, float* lse, void* workspace, size_t workspace_bytes,
                        void* stream);

/*
 * Speculative verify: n_q in 1..4 new positions per sequence, causal among themselves
 * ("Scaling Kimi K3 ...", section "并行度必须适配真正的形状": four verify positions per
 * sequence). n_q = 1 is exactly mla_decode.
 *   q    device, [B][n_q][H][576] bfloat16
 *   out  device, [B][n_q][H][512] bfloat16
 *   lse  device, [B][n_q][H] float32, or NULL
 */
mla_status_t mla_verify(const mla_kv_t* kv, const void* q, int B, int n_q, int H,
                        float sm_scale, void* out, float* lse, void* workspace,
                        size_t workspace_bytes, void* stream);

/*
 * mla_verify with a float32 output: the normalised attention output over the keys that kv
 * describes, not rounded to bfloat16, for results that are merged afterwards. In
 * decode-context parallelism every rank holds a shard of each sequence's positions, attends
 * to its shard alone, and the shards' outputs are combined through their log-sum-exp
 * ("Scaling Kimi K3 on AMD Instinct MI355X: Matching NVIDIA HGX B300 Throughput per GPU on
 * AgentX", section "缓存可复用，还要能一致地恢复"); keeping the shard outputs in float32
 * leaves a single bfloat16 rounding, in mla_merge_lse. Arguments, workspace, masking and
 * errors as mla_verify (workspace from mla_workspace_size(MLA_OP_VERIFY, ...)), except:
 *   out  device, [B][n_q][H][512] float32 (16-byte aligned)
 * A sequence with no key gives out = 0 and lse = -inf, which mla_merge_lse weighs as 0.
 */
mla_status_t mla_verify_f32(const mla_kv_t* kv, const void* q, int B, int n_q, int H,
                            float sm_scale, float* out, float* lse, void* workspace,
                            size_t workspace_bytes, void* stream);

/*
 * mla_verify_f32 over one rank's shard of the positions, with the causal limit moved:
 * key n of the view (0-based within it) is visible to new position j iff
 * n <= seq_lens[b] - n_q + j + visible_shift. Under decode-context parallelism ("Scaling
 * Kimi K3 ...", section "缓存可复用，还要能一致地恢复") the n_q new positions sit in the last
 * shard of a sequence; every other shard lies wholly before them, so all of its keys are
 * visible to all n_q positions: visible_shift >= n_q - 1 says so (values above n_q - 1
 * act as n_q - 1), and each page of the shard is read once for the n_q positions
 * together. visible_shift = 0 is mla_verify_f32. Negative: MLA_ERR_INVALID_ARG.
 * Arguments, workspace and errors otherwise as mla_verify_f32.
 */
mla_status_t mla_verify_f32_shard(const mla_kv_t* kv, const void* q, int B, int n_q, int H,
                                  float sm_scale, int visible_shift, float* out, float* lse,
                                  void* workspace, size_t workspace_bytes, void* stream);

/*
 * Causal chunked prefill of one sequence: T new positions attend to the cached prefix
 * and causally to each other ("AMD MI355X推理Kimi K3：吞吐量超NVIDIA，首字优化显著",
 * section "首Token等待优化：简单补零解决大问题": long cold prefill through the MLA
 * prefill kernel). kv describes one sequence (seq_lens[0] = prefix + T).
 *   q    device, [T][H][576] bfloat16
 *   out  device, [T][H][512] bfloat16
 *   lse  device, [T][H] float32, or NULL
 * Blocks of 48 / H positions go to the SMs a round at a time, longest first. When the
 * last round would leave SMs idle, its blocks run as a second kernel over their keys'
 * two halves and a third kernel merges the halves (the workspace holds their partials):
 * one launch or three, all on `stream`.
 */
mla_status_t mla_prefill(const mla_kv_t* kv, const void* q, int T, int H, float sm_scale,
                         void* out, float* lse, void* workspace, size_t workspace_bytes,
                         void* stream);

/*
 * Causal prefill of one sequence in the MHA (non-absorbed) form. Keys and values of every
 * head are up-projected from the shared latent ("MI355X Kimi K2.5 vLLM AITER 7x speedup",
 * section "PR #35850 修复了什么": K and V come from one compressed latent): for head h and
 * cached position n, key = [c_n W_UK_h ; r_n] (192 wide) and value = c_n W_UV_h (128 wide),
 * c_n the 512-wide latent and r_n the 64 RoPE dims of the row, dequantised under
 * kv->kv_scale. New position t (of the last T of L cached) sees keys n <= L - T + t; scores
 * are q . key x sm_scale. The tensor cores see the up-projected keys as a bf16 pair (high
 * and low parts: about 16 significant bits), the RoPE part exactly, and the values and the
 * probabilities in fp16, so the results meet the same tolerances as mla_prefill.
 *   kv     the cache (page size a multiple of 64); kv->seq_lens is not read: L is given
 *          on the host because it sizes the up-projection; sequence 0 of the page table
 *   L      cached positions including the T new ones, 1 <= T <= L <= page-table capacity
 *   q      device, [T][H][192] bfloat16 (128 no-RoPE dims, then 64 RoPE dims), 16-B aligned
 *   w_ukv  device, [512][H][256] bfloat16: for head h, columns 0..127 are W_UK_h and
 *          128..255 are W_UV_h
 *   out    device, [T][H][128] bfloat16, 16-B aligned
 *   lse    device, [T][H] float32 (natural log), or NULL
 *   workspace  device, 256-B aligned, mla_prefill_mha_workspace_size(L, H, device) bytes:
 *          the dequantised latent, the up-projected keys and values, status words.
 * Errors as mla_prefill; a page index outside the pool is reported by mla_read_status.
 * Launches: a dequantisation kernel, the up-projection GEMM (tcgen05), the attention kernel
 * (and a merge of key-split units when the last round of units is cut along the keys).
 */
size_t mla_prefill_mha_workspace_size(int L, int H, int device);
mla_status_t mla_prefill_mha(const mla_kv_t* kv, int L, const void* q, int T, int H,
                             const void* w_ukv, float sm_scale, void* out, float* lse,
                             void* workspace, size_t workspace_bytes, void* stream);

/*
 * mla_prefill_mha with every tensor-core operand in bfloat16: keys (x kv_scale), values and
 * probabilities are each rounded to bf16 once, as a plain bf16 flash-attention prefill
 * would. It moves 80 KB per 128 keys instead of 112 KB and runs about a fifth faster, but
 * those three roundings make it miss mla_prefill's tolerances: relative L2 up to about
 * 3e-3 and LSE errors up to about 4e-3 x max(1, |lse|) on rows that see few keys.
 * Arguments, workspace and errors as mla_prefill_mha.
 */
mla_status_t mla_prefill_mha_bf16(const mla_kv_t* kv, int L, const void* q, int T, int H,
                                  const void* w_ukv, float sm_scale, void* out, float* lse,
                                  void* workspace, size_t workspace_bytes, void* stream);

/*
 * Log-sum-exp merge of S partial results per row ("Scaling Kimi K3 ...", section
 * "缓存可复用，还要能一致地恢复"): lse = ln sum_s exp(lse_s),
 * out = sum_s exp(lse_s - lse) * out_s. Partials with lse_s = -inf carry weight 0; a row
 * whose partials are all -inf gets out = 0, lse = -inf.
 *   part_out  device, [S][R][512] float32 (each partial already normalised)
 *   part_lse  device, [S][R] float32 (natural log)
 *   out       device, [R][512] bfloat16
 *   lse       device, [R] float32, or NULL
 * This is the step a position-sharded (DCP) deployment runs after gathering partials.
 */
mla_status_t mla_merge_lse(const float* part_out, const float* part_lse, int S, int64_t R,
                           void* out, float* lse, void* stream);

/*
 * Append new latent rows to the paged cache ("MI355X Kimi K2.5 vLLM AITER 7x speedup",
 * section "PR #35850 修复了什么": the FP8 KV cache handled natively; "Scaling Kimi K3 ...",
 * section "缓存可复用，还要能一致地恢复": 576 FP8 bytes per position). For every i < n with
 * slots[i] >= 0, cache row slots[i] (page slots[i] / page_size, position slots[i] %
 * page_size) becomes the e4m3 codes of x_i * (1 / kv_scale): the reciprocal and each
 * product are rounded to binary32, the conversion rounds to nearest even and saturates
 * finite values and infinities at +-448 (NaN stays NaN); this is also how the library's
 * input generator quantises the rows it draws. Rows with a negative slot are skipped
 * (padding).
 *   pool    device, [num_pages][page_size][576] e4m3 codes, 16-byte aligned (written)
 *   x       device, [n][576] bfloat16, 16-byte aligned
 *   slots   device, [n] int64 flat cache rows, 8-byte aligned
 *   kv_scale the cache's per-tensor scale (> 0, finite)
 *   status  device word or NULL: set to MLA_ERR_BOUNDS (if it held 0) when a slot is not
 *           below num_pages * page_size; that row is not written
 * Rows are written in no particular order: two rows with the same slot leave one of them.
 */
mla_status_t mla_cache_append(uint8_t* pool, int64_t num_pages, int32_t page_size,
                              const void* x, const int64_t* slots, int64_t n, float kv_scale,
                              unsigned* status, void* stream);

/*
 * Top-k renormalisation of probability rows, the sampling step of speculative-verify
 * acceptance ("MI355X Kimi K2.5 vLLM AITER 7x speedup": top_k_renorm_prob among the
 * serving stack's sampling kernels). Per row r with k_r = top_k ? top_k[r] : k:
 * pivot = the k_r-th largest probability; every p >= pivot is kept (ties at the pivot
 * included), out = p / (sum of the kept entries), the rest 0. k_r <= 0 or k_r >= V keeps
 * the whole row. Probabilities must be non-negative and finite.
 *   probs  device, [B][V] float32 (read)
 *   out    device, [B][V] float32 (written; may not alias probs)
 *   top_k  device, [B] int32, or NULL to use k for every row
 */
mla_status_t mla_top_k_renorm_prob(const float* probs, float* out, int B, int V,
                                   const int32_t* top_k, int k, void* stream);

/*
 * Synchronises `stream`, then returns the status the last call on this workspace left
 * (MLA_OK, MLA_ERR_BOUNDS or MLA_ERR_TIMEOUT: the first non-zero of the words its CTAs
 * wrote at exit), or MLA_ERR_CUDA if the stream itself reports an error.
 */
mla_status_t mla_read_status(const void* workspace, size_t workspace_bytes, void* stream);

/*
 * Test hook for the failure path: the next mla_decode / mla_verify / mla_verify_f32 call on
 * this thread launches its attention kernel with the key loads switched off, so every wait
 * on them gives up after its limit (about a second) and the call's status words report
 * MLA_ERR_TIMEOUT; the kernel still returns, the context stays usable, and the outputs of
 * that call are undefined. Not for production use.
 */
void mla_test_stall_next_call(void);

/* Static, human-readable name of a status code. */
const char* mla_status_string(mla_status_t status);

/* Number of kernel launches the last compute call on this host thread enqueued. */
int mla_last_launch_count(void);

/*
 * Profiling hook. When both are non-NULL, the next compute calls on this host thread
 * record `start` (a cudaEvent_t passed as void*) on their stream just before the main
 * attention kernel and `stop` just after it, so cudaEventElapsedTime() gives that
 * kernel's own duration. Pass NULL, NULL to switch it off. The events stay owned by the
 * caller.
 */
void mla_set_profile_events(void* start, void* stop);

/*
 * Profiling hook. With a device buffer of `bytes` (8-byte aligned), the next decode /
 * verify / prefill calls on this host thread make each CTA c of their attention kernel
 * (while c < bytes / 128) write sixteen 64-bit words at buffer + 128 c: the GPU's global
 * timer (ns) at entry, after the wait on the previous kernel, after the split plan and the
 * first tile loads issued, when the first tile's scores were read, when the last tile's
 * probabilities were written, when the last values MMA completed, after its last epilogue
 * and at exit; then (tiles << 32 | units) it processed; then, for CTAs with two units or
 * more, the end of the first unit's epilogue and the second unit's first scores; then
 * (decode / verify) the end of the plan's scan and the end of its L2 prefetches (words 13-15
 * are not written). NULL switches
 * it off. The buffer stays owned by the caller; the results are undefined while two calls
 * overlap on the GPU.
 */
void mla_set_trace_buffer(void* device_buffer, size_t bytes);

/*
 * Decode without a caller-provided workspace. (The pages describe no such entry point; it
 * exists for callers of this library that cannot allocate device memory: an engine that
 * has already reserved nearly all device memory for its own pools, or a latency-critical
 * loop where cudaMalloc/cudaFree, which can synchronise the device, are not allowed.)
 *
 * Same arguments, layouts and results as mla_decode, but the workspace is a fixed array
 * of MLA_STATIC_WS_BYTES owned by the library in device memory: every GPU on which the
 * library's kernels are loaded holds it until the process exits. No memory is allocated
 * by this call.
 *  - A call whose mla_workspace_size(MLA_OP_DECODE, B, H, 1, device) exceeds
 *    MLA_STATIC_WS_BYTES is rejected with MLA_ERR_WORKSPACE before anything is enqueued.
 *    The decode workspace grows with H and the SM count, not with B: 16 MiB covers
 *    16-head decode of any batch on a 152-SM GB300 (the partial outputs and staged query
 *    rows take about 13 MB of it).
 *  - The first call on each device (and the first after the device's context changed,
 *    for instance after cudaDeviceReset) looks up the array's device address (a runtime
 *    symbol query); make that first call outside any CUDA stream capture.
 *  - All calls on a device share the one array, which keeps the previous call's
 *    contents (each call rewrites everything it reads). Calls whose work overlaps on
 *    the GPU (different streams without ordering,
 *    or several host threads) race on it and give wrong results: serialise them.
 *  - The device-side status words of these calls (MLA_ERR_BOUNDS, MLA_ERR_TIMEOUT) are
 *    read with mla_read_status_static.
 */
#define MLA_STATIC_WS_BYTES (16u << 20)
mla_status_t mla_decode_static_ws(const mla_kv_t* kv, const void* q, int B, int H,
                                  float sm_scale, void* out, float* lse, void* stream);

/*
 * mla_read_status for the library-owned workspace of mla_decode_static_ws on the current
 * device: synchronises `stream`, then returns the status the last mla_decode_static_ws
 * call on this device left (MLA_OK, MLA_ERR_BOUNDS or MLA_ERR_TIMEOUT), or MLA_ERR_CUDA.
 * Allocates nothing. (No counterpart on the pages, like mla_decode_static_ws.)
 */
mla_status_t mla_read_status_static(void* stream);

#ifdef __cplusplus
}
#endif
#endif /* MLA_H */
