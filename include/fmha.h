/*
 * fmha.h -- C ABI of the GB300 (sm_103a) fused multi-head attention forward.
 *
 *   O = softmax(scale * Q K^T + mask) V      (per batch, query head)
 *   LSE = log(sum_j exp(scale * q.k_j))      (natural log, visible keys only)
 *
 * computed with an online (running max / running sum) softmax so that the
 * score and probability matrices never leave the chip.
 *
 * Passages that define the operation (page title, section):
 *  - "fmha sm120 : 超越 torch.sdpa(flash-attention-2)", §1 flash attention:
 *    MHA = softmax(q @ k^T * scale) @ v on [batch, seq, heads, head_dim]
 *    tensors, O shaped like Q, scale conventionally 1/sqrt(head_dim); §2:
 *    grouped-query attention maps query head h to kv head h / (H / H_k).
 *  - "FMHA for Blackwell: Forward" (CUTLASS example 77 README): head dims
 *    32/64/128, fp8/fp16/bf16 inputs.
 *  - "CUTLASS Blackwell FMHA 示例完全解析": §融合扩展点 (masks: none, residual,
 *    causal with q-begin / q-end alignment, masked scores are -infinity);
 *    §变长序列 (cumulative lengths, total_length, a padding batch ahead of the
 *    packed data); §验证机制 (O and LSE are both outputs); §核心设计 (the
 *    output scale is applied in fp32 before the cast to the output type).
 *
 * All functions are thread-safe.  Nothing here allocates device memory except
 * one lazily created 4-byte device status word per library instance.
 */
#ifndef FMHA_H
#define FMHA_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>   /* cudaStream_t */

#ifdef __cplusplus
extern "C" {
#endif

/* Storage types of Q, K, V and O. */
enum fmha_dtype {
    FMHA_F16 = 0,   /* IEEE binary16 */
    FMHA_BF16 = 1,  /* bfloat16 */
    FMHA_E4M3 = 2   /* OCP fp8 E4M3 ("fn": no inf, max 448) */
};

/* A device buffer and its storage type. */
typedef struct fmha_tensor {
    void *data;
    int dtype;      /* enum fmha_dtype */
} fmha_tensor;

enum fmha_mask {
    FMHA_MASK_NONE = 0,      /* every key of the sequence is visible */
    FMHA_MASK_RESIDUAL = 1,  /* same result as NONE: keys >= Sk are dropped */
    FMHA_MASK_CAUSAL = 2     /* key j visible to query i iff j <= i + offset */
};

enum fmha_causal_type {
    FMHA_CAUSAL_QBEGIN = 0,  /* offset 0: queries aligned to the first key */
    FMHA_CAUSAL_QEND = 1     /* offset Sk - Sq: last query sees every key */
};

enum fmha_status {
    FMHA_OK = 0,
    FMHA_ERR_INVALID_ARG = -1,   /* bad pointer, size, enum or varlen arguments */
    FMHA_ERR_UNSUPPORTED = -2,   /* valid but not supported: dtype combination,
                                    alignment, device not sm_103 */
    FMHA_ERR_CUDA = -3,          /* a CUDA runtime / driver call failed */
    FMHA_ERR_TIMEOUT = -4        /* a bounded on-device wait expired
                                    (reported by fmha_device_status) */
};

/*
 * fmha_fwd -- fused attention forward on the tcgen05 tensor cores.
 *
 * Arguments
 *   q, k, v      inputs.  k and v have q's dtype.
 *   o            output.  dtype == q's for fp16/bf16; FMHA_E4M3 (saturating
 *                round-to-nearest-even) for e4m3 inputs.
 *   lse          fp32 log-sum-exp output, or NULL to skip it.
 *   B            batch size (number of sequences when varlen).
 *   H, H_k       query heads and key/value heads; H % H_k == 0 (GQA, MQA
 *                when H_k == 1).  Query head h reads kv head h / (H / H_k).
 *   Sq, Sk       query and key lengths (fixed-length mode; ignored if varlen).
 *   D            head dim: 32, 64 or 128.
 *   scale        softmax scale applied to Q K^T (1/sqrt(D) is the usual);
 *                finite and > 0, otherwise FMHA_ERR_INVALID_ARG.
 *   out_scale    fp32 factor applied to O before the cast to o's dtype.
 *                It does not enter LSE.
 *   mask         enum fmha_mask.  causal_type: enum fmha_causal_type.
 *   cu_seqlens_q, cu_seqlens_k
 *                both NULL: fixed length.  Both non-NULL: variable length,
 *                int32 device arrays of B+1 non-decreasing entries starting
 *                at 0; sequence b owns packed q rows [cu_q[b], cu_q[b+1]) and
 *                k/v rows [cu_k[b], cu_k[b+1]).  One NULL: INVALID_ARG.
 *   max_len      varlen: >= every per-sequence q and k length.
 *   total_length varlen: number of rows allocated in every packed tensor,
 *                >= cu_q[B] and >= cu_k[B].  It bounds every load.
 *   stream       CUDA stream; the call is asynchronous on it.
 *
 * Layouts (all contiguous, row-major):
 *   fixed:  q, o [B, Sq, H, D];  k, v [B, Sk, H_k, D];  lse [B, H, Sq]
 *   varlen: q, o [total_length, H, D];  k, v [total_length, H_k, D];
 *           lse [H, total_length]; each pointer addresses the first packed row.
 *   Varlen callers keep one batch of valid padding rows ahead of the packed
 *   data (the layout of the CUTLASS example); this library never reads or
 *   writes it, and never writes o or lse rows outside [0, cu_q[B]).
 *   Input rows that share a load tile with a sequence but lie outside it are
 *   read and then masked, so inputs must hold no NaN or Inf.
 *
 * Semantics: a query row with no visible key (causal q-end with Sq_b > Sk_b
 * rows, or Sk_b == 0) gets O = 0 and LSE = -infinity.
 *
 * Ownership: the caller owns every buffer; the library keeps no pointer after
 * the call returns.  Data pointers must be 16-byte aligned (TMA), otherwise
 * FMHA_ERR_UNSUPPORTED.
 *
 * Errors: arguments are validated before anything is launched; on error
 * nothing is launched and the status says why.  Returns FMHA_OK when the work
 * was enqueued (or there was nothing to do).
 */
int fmha_fwd(fmha_tensor q, fmha_tensor k, fmha_tensor v, fmha_tensor o, float *lse,
             int B, int H, int H_k, int Sq, int Sk, int D,
             float scale, float out_scale, int mask, int causal_type,
             const int *cu_seqlens_q, const int *cu_seqlens_k, int max_len,
             int64_t total_length, cudaStream_t stream);

/*
 * fmha_fwd_simt -- the same operation on CUDA cores (fp32 FMA, no tensor
 * cores).  Same arguments, layouts, semantics and errors as fmha_fwd.  It is
 * a slow cross-check of the tensor-core kernel, not a fast path.
 */
int fmha_fwd_simt(fmha_tensor q, fmha_tensor k, fmha_tensor v, fmha_tensor o, float *lse,
                  int B, int H, int H_k, int Sq, int Sk, int D,
                  float scale, float out_scale, int mask, int causal_type,
                  const int *cu_seqlens_q, const int *cu_seqlens_k, int max_len,
                  int64_t total_length, cudaStream_t stream);

/*
 * fmha_fwd_splitkv -- fmha_fwd with every work unit's key range cut into
 * num_splits contiguous pieces, for shapes with few (batch, head, 256-row
 * query block) units and long key sequences, where fmha_fwd would leave most
 * SMs idle.  Each piece writes a normalised fp32 partial O and its LSE into
 * the workspace; a second kernel merges them exactly:
 *   LSE = ln sum_s exp(LSE_s),   O = out_scale * sum_s exp(LSE_s - LSE) * O_s.
 * ("CUTLASS Blackwell FMHA 示例完全解析", §MLA 与 split-KV、reduction 策略: the
 * same split-KV reduction, there for MLA decoding.)
 *
 * Arguments as fmha_fwd, plus:
 *   num_splits       1..256.  More splits than key tiles leave some pieces
 *                    empty (they contribute nothing).
 *   workspace        device scratch owned by the caller, 256-byte aligned,
 *                    at least fmha_fwd_splitkv_workspace_size(...) bytes.  Its
 *                    contents on entry do not matter; every byte the merge
 *                    reads is written first in the same call.  Two calls that
 *                    share a workspace must not overlap on the GPU.
 *   workspace_bytes  its size.
 * Errors: as fmha_fwd; FMHA_ERR_INVALID_ARG for num_splits out of range or a
 * missing, misaligned or too small workspace.  Two kernels are enqueued on
 * stream; o and lse are complete when the second one finishes.
 */
int fmha_fwd_splitkv(fmha_tensor q, fmha_tensor k, fmha_tensor v, fmha_tensor o, float *lse,
                     int B, int H, int H_k, int Sq, int Sk, int D,
                     float scale, float out_scale, int mask, int causal_type,
                     const int *cu_seqlens_q, const int *cu_seqlens_k, int max_len,
                     int64_t total_length, int num_splits, void *workspace,
                     size_t workspace_bytes, cudaStream_t stream);

/*
 * Workspace bytes fmha_fwd_splitkv needs.  Fixed length: pass total_length = 0
 * (rows = B * Sq).  Variable length: pass the call's total_length (rows =
 * total_length; B and Sq are then ignored).  Returns 0 for invalid arguments.
 */
size_t fmha_fwd_splitkv_workspace_size(int B, int H, int Sq, int D, int num_splits,
                                       int64_t total_length);

/*
 * fmha_fwd_splitkv_noalloc -- fmha_fwd_splitkv for callers that must not
 * allocate device memory while they run: processes that reserve their HBM
 * once at start-up and treat a later cudaMalloc as a failure (it can fail,
 * fragment the reservation or stall the device), or plug-ins whose host
 * framework owns every device allocation.  The pages have no counterpart of
 * this entry point.
 *
 * Same arguments as fmha_fwd_splitkv without workspace / workspace_bytes:
 * the scratch is a library-owned device array of FMHA_NOALLOC_SCRATCH_BYTES
 * (32 MiB), reserved on every GPU that loads the library until the process
 * exits.  The caller still owns q, k, v, o and lse.  No device memory is
 * allocated or freed by this call.
 *
 * - Every call looks up the array's device address in the current context, a
 *   host-side step (the first call on a device also loads the library's device
 *   code there); make the first call on a device before any stream capture.
 * - Arguments are checked first, exactly as fmha_fwd_splitkv checks them: an
 *   empty problem returns FMHA_OK and a bad argument its own status.  Then
 *   problems whose split-KV scratch (fmha_fwd_splitkv_workspace_size) exceeds
 *   the array return FMHA_ERR_UNSUPPORTED without launching; use
 *   fmha_fwd_splitkv with a workspace for those.
 * - Every call uses the same array.  Nothing in it needs to start at zero
 *   (each call writes every byte it later reads), but two calls whose kernels
 *   overlap on the GPU -- on different streams, or different host threads --
 *   race on it and corrupt each other's results.  Serialise them (one stream).
 * Errors otherwise as fmha_fwd_splitkv.
 */
#define FMHA_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
int fmha_fwd_splitkv_noalloc(fmha_tensor q, fmha_tensor k, fmha_tensor v, fmha_tensor o, float *lse,
                             int B, int H, int H_k, int Sq, int Sk, int D,
                             float scale, float out_scale, int mask, int causal_type,
                             const int *cu_seqlens_q, const int *cu_seqlens_k, int max_len,
                             int64_t total_length, int num_splits, cudaStream_t stream);

/*
 * fmha_gen_fwd -- generation phase: one new query token per sequence attends
 * to that sequence's entry of a key/value cache ("CUTLASS Blackwell FMHA
 * 示例完全解析", §FMHA for Blackwell 生成阶段: KV-cache forward with batch
 * index remapping, cache-only mode and per-entry sequence lengths; head dim
 * 128; one query-head group per thread block).
 *
 * For sequence b, query head h, kv head g = h / (H / H_k), cache entry
 * e = batch_idx ? batch_idx[b] : b and L = seqlen[b] cached tokens:
 *   keys   = K_cache[e, 0..L-1, g, :], then (insert mode) K_new[b, g, :]
 *   values = V_cache[e, 0..L-1, g, :], then (insert mode) V_new[b, g, :]
 *   O[b, h, :] = out_scale * softmax(scale * q[b, h, :] . keys) values
 *   lse[b, h]  = natural-log log-sum-exp of the scaled scores
 * (no key at all: O = 0, lse = -inf).  In insert mode (k_new.data and
 * v_new.data both non-NULL) the call also writes K_new[b, g, :] and
 * V_new[b, g, :] into row L of entry e of the caches; it does not change
 * seqlen (the caller advances it).  Cache-only mode (both NULL) neither
 * reads nor writes new rows.
 *
 * Layouts (contiguous, device memory):
 *   q, o               [B, H, 128]
 *   k_cache, v_cache   [B_cache, S_max, H_k, 128]
 *   k_new, v_new       [B, H_k, 128]
 *   seqlen, batch_idx  int32 [B] (batch_idx may be NULL: entry b)
 *   lse                float [B, H], or NULL
 * All tensors share one dtype, FMHA_F16, FMHA_BF16 or FMHA_E4M3; D must be
 * 128 and H / H_k at most 32.  Device pointers must be 16-byte aligned.  With
 * e4m3 the weights P are rounded to e4m3 before P.V (their row sum is not),
 * and O is rounded to e4m3 with saturation.
 * Requirements the host cannot check (they live in device memory):
 * 0 <= seqlen[b] <= S_max - (insert ? 1 : 0) and 0 <= batch_idx[b] < B_cache;
 * a kernel that meets a violation clamps the length (and inserts nothing) or
 * reads zeros for the missing entry, and fmha_device_status then reports
 * FMHA_ERR_INVALID_ARG.  In insert mode two sequences must not share an entry.
 * Cached rows at or past a sequence's length are never used, and may hold any
 * bits, including NaN.
 *
 * workspace: caller-owned scratch of at least fmha_gen_workspace_size(...)
 * bytes, 256-byte aligned; nothing in it needs initialising; it must not be
 * shared with a call that may run concurrently.  The call allocates nothing
 * and is asynchronous on `stream` (a kernel, then a merge kernel).
 * Returns FMHA_OK, FMHA_ERR_INVALID_ARG (bad sizes or pointers, scale not
 * finite and > 0, workspace too small or misaligned, only one of k_new /
 * v_new), FMHA_ERR_UNSUPPORTED (dtype, alignment) or FMHA_ERR_CUDA.
 * B = 0 succeeds without a launch.
 */
int fmha_gen_fwd(fmha_tensor q, fmha_tensor k_cache, fmha_tensor v_cache,
                 fmha_tensor k_new, fmha_tensor v_new, fmha_tensor o, float *lse,
                 int B, int H, int H_k, int D, int B_cache, int S_max,
                 const int *seqlen, const int *batch_idx, float scale, float out_scale,
                 void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Workspace bytes fmha_gen_fwd needs for these sizes: an fp32 partial O row
 * and LSE per (sequence, query head, key chunk), at most one chunk per key
 * tile of S_max plus one (tiles of 64 keys when H_k is even and H / H_k <= 16,
 * else 128).  0 for invalid sizes.
 */
size_t fmha_gen_workspace_size(int B, int H, int H_k, int D, int S_max);

/*
 * fmha_bwd -- backward pass of fmha_fwd: dQ, dK, dV from dO ("CUTLASS
 * Blackwell FMHA 示例完全解析", §FMHA for Blackwell 反向 (Backward): row sums
 * of O * dO, a dK/dV kernel and a dQ kernel, Q and K blocking 128, causal
 * masking, head dims 64 and 128, no GQA).
 *
 * With P = softmax(scale Q K^T + mask) (the forward's definition, out_scale
 * = 1) and a loss whose gradient with respect to O is dO:
 *   dV = P^T dO,  dS = P * (dO V^T - rowsum(dO * O)),  dQ = scale dS K,
 *   dK = scale dS^T Q.
 * Inputs: q, o, dout [B, Sq, H, D]; k, v [B, Sk, H, D] (H_k = H: no GQA);
 * lse float [B, H, Sq] as written by fmha_fwd for the same q, k, v, mask.
 * Outputs: dq [B, Sq, H, D], dk, dv [B, Sk, H, D].  Dtypes: all FMHA_F16 or
 * all FMHA_BF16; or e4m3 inputs (q, k, v, o, dout FMHA_E4M3, as fmha_fwd
 * writes o for e4m3) with FMHA_BF16 gradients.  The page lists fp8 among the
 * backward's types but states no scaling of P, dS or the gradients; without
 * scales, rounding dS to e4m3 would flush most of it (|dS| is often below
 * e4m3's smallest subnormal, 2^-9), so e4m3 inputs are widened exactly to
 * bf16 in the workspace and the products run on the bf16 path.  D is 64 or
 * 128; mask NONE, RESIDUAL or CAUSAL (q-begin or q-end), as fmha_fwd.  Fixed
 * length only.  Tensors 16-byte aligned, lse 4-byte aligned.
 * workspace: caller-owned, fmha_bwd_workspace_size_ex(B, H, Sq, Sk, D,
 * q.dtype) bytes (for 16-bit types equal to fmha_bwd_workspace_size(B, H,
 * Sq)), 256-byte aligned (two fp32 values per query row, -LSE*log2(e) and
 * -dO.O, each row padded to a multiple of 128; for e4m3 then the bf16 copies
 * of q, o, dout, k and v); no initialisation needed; not shared with a
 * concurrent call.  Asynchronous on `stream` (three kernels, four for e4m3);
 * allocates nothing.  Returns FMHA_OK, FMHA_ERR_INVALID_ARG (sizes, scale, mask,
 * pointers, workspace), FMHA_ERR_UNSUPPORTED (dtype, alignment) or
 * FMHA_ERR_CUDA.  B = 0 succeeds without a launch; Sq = 0 or Sk = 0 clears
 * the gradients that exist.
 */
int fmha_bwd(fmha_tensor q, fmha_tensor k, fmha_tensor v, fmha_tensor o, fmha_tensor dout,
             const float *lse, fmha_tensor dq, fmha_tensor dk, fmha_tensor dv,
             int B, int H, int Sq, int Sk, int D, float scale, int mask, int causal_type,
             void *workspace, size_t workspace_bytes, cudaStream_t stream);

/* Workspace bytes fmha_bwd needs for 16-bit inputs (0 for invalid sizes). */
size_t fmha_bwd_workspace_size(int B, int H, int Sq);

/* Workspace bytes fmha_bwd needs for inputs of type `dtype` (FMHA_F16,
 * FMHA_BF16 or FMHA_E4M3); 0 for invalid sizes or another dtype. */
size_t fmha_bwd_workspace_size_ex(int B, int H, int Sq, int Sk, int D, int dtype);

/* Text for a status code (static storage, never NULL). */
const char *fmha_status_string(int status);

/*
 * fmha_device_status -- read the device-side status word of the current
 * device: FMHA_OK, FMHA_ERR_TIMEOUT if a kernel gave up a bounded wait
 * (it then skipped its remaining work and released its resources), or
 * FMHA_ERR_INVALID_ARG if fmha_gen_fwd met a sequence length or cache entry
 * outside its bounds.
 * Synchronises the device.  reset != 0 clears the word.  Returns
 * FMHA_ERR_CUDA if the word cannot be read.
 */
int fmha_device_status(int reset);

/*
 * fmha_set_wait_limit_ns -- test hook for the failure path of fmha_fwd,
 * fmha_fwd_splitkv, fmha_gen_fwd and fmha_bwd: their bounded on-device waits
 * give up after ns nanoseconds instead of 4 s (ns = 0 restores 4 s).  A wait
 * that expires records FMHA_ERR_TIMEOUT for fmha_device_status and makes the
 * call's CTAs stop issuing work, wait (bounded) for the copies and MMAs they
 * have in flight, free their tensor memory and exit; the outputs of that call
 * are then undefined and the context stays usable.  Applies to launches that
 * start after the call returns.  Returns FMHA_OK or FMHA_ERR_CUDA.
 */
int fmha_set_wait_limit_ns(unsigned long long ns);

/*
 * fmha_set_test_gate -- test hook: while on (on != 0), the producer warp of
 * every fmha_fwd / fmha_fwd_splitkv CTA, of every fmha_gen_fwd attention CTA
 * and of every fmha_bwd dQ and dK/dV CTA first waits for a device flag that
 * nothing sets, so that bounded wait expires after the limit of
 * fmha_set_wait_limit_ns and the launch takes the failure path above before
 * any copy is issued.  Off by default.  Returns FMHA_OK or FMHA_ERR_CUDA.
 */
int fmha_set_test_gate(int on);

/*
 * fmha_kv_tile_range -- host copy of the scheduler's key-tile bounds for one
 * query tile (exposed for testing).  For query rows [q_row0, q_row0 + q_rows)
 * of a sequence with Sq queries and Sk keys, key tiles of tile_n rows:
 *   *n_tiles    = number of key tiles that hold at least one visible key,
 *   *n_unmasked = leading key tiles in which every key is visible to every
 *                 query row of the tile (no mask needs to be applied there).
 * Rows at or past Sq are ignored.  Returns FMHA_OK or FMHA_ERR_INVALID_ARG.
 * ("CUTLASS Blackwell FMHA 示例完全解析", §融合扩展点: get_trip_count,
 * get_masked_trip_count, get_unmasked_trip_count.)
 */
int fmha_kv_tile_range(int q_row0, int q_rows, int Sq, int Sk, int mask, int causal_type,
                       int tile_n, int *n_tiles, int *n_unmasked);

#ifdef __cplusplus
}
#endif
#endif /* FMHA_H */
