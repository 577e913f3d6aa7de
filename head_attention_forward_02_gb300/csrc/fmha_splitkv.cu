// fmha_splitkv.cu -- split-KV attention forward: the tensor-core kernel run
// over key ranges, then an LSE-weighted merge of the partial results.
//
// For shapes with few (batch, head, query block) units and long keys, most
// SMs would idle.  Cutting each unit's key tiles into S contiguous ranges
// gives S times as many work items.  Range s yields a normalised partial
// O_s = sum_j p_j V_j / l_s and LSE_s = ln l_s (both relative to the same
// scores), so the exact result is
//     LSE = ln sum_s exp(LSE_s),   O = out_scale * sum_s exp(LSE_s - LSE) O_s
// -- the same merge as the split-KV reduction of the CUTLASS MLA example
// ("CUTLASS Blackwell FMHA 示例完全解析", §MLA 与 split-KV、reduction 策略),
// written here for the forward kernel.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <math.h>

#include "fmha_common.h"

namespace fmha {
namespace {

constexpr int kMaxSplits = 256;
constexpr int kCombineWarps = 8;

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

template <int PER>
__device__ __forceinline__ void load_f(const float *p, float (&x)[PER]) {
    if constexpr (PER == 4) {
        const float4 v = *reinterpret_cast<const float4 *>(p);
        x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
    } else if constexpr (PER == 2) {
        const float2 v = *reinterpret_cast<const float2 *>(p);
        x[0] = v.x; x[1] = v.y;
    } else {
        x[0] = p[0];
    }
}

template <int PER>
__device__ __forceinline__ void store_o(void *base, int64_t idx, int dtype, const float (&x)[PER]) {
    if (dtype == FMHA_BF16) {
        __nv_bfloat16 *o = reinterpret_cast<__nv_bfloat16 *>(base) + idx;
#pragma unroll
        for (int i = 0; i < PER; ++i) o[i] = __float2bfloat16_rn(x[i]);
    } else if (dtype == FMHA_F16) {
        __half *o = reinterpret_cast<__half *>(base) + idx;
#pragma unroll
        for (int i = 0; i < PER; ++i) o[i] = __float2half_rn(x[i]);
    } else {
        __nv_fp8_storage_t *o = reinterpret_cast<__nv_fp8_storage_t *>(base) + idx;
#pragma unroll
        for (int i = 0; i < PER; ++i) o[i] = __nv_cvt_float_to_fp8(x[i], __NV_SATFINITE, __NV_E4M3);
    }
}

// One warp per (query row, head): merge the num_splits partial results.
template <int D>
__global__ void __launch_bounds__(kCombineWarps * 32) combine_kernel(const Params p) {
    constexpr int PER = D / 32;
    const int lane = threadIdx.x & 31;
    const int64_t item = (int64_t)blockIdx.x * kCombineWarps + (threadIdx.x >> 5);
    const int64_t rows = p.varlen ? (int64_t)p.cu_q[p.B] : (int64_t)p.B * p.Sq;
    if (item >= rows * p.H) return;
    const int64_t row = item / p.H;
    const int h = (int)(item - row * p.H);
    const int ns = p.num_splits;
    const int64_t split_stride = p.part_rows * p.H;          // elements between splits of part_lse
    // the partials are the attention kernel's: wait for it (and its memory)
    // here; the launch and the lines above overlap its tail
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const float *plse = p.part_lse + row * p.H + h;
    float m = -INFINITY;
    for (int s = lane; s < ns; s += 32) m = fmaxf(m, plse[s * split_stride]);
    m = warp_max(m);
    float acc[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) acc[i] = 0.f;
    float den = 0.f;
    if (m != -INFINITY) {
        const float *po = p.part_o + (row * p.H + h) * D + lane * PER;
        for (int s = 0; s < ns; ++s) {
            const float ls = plse[s * split_stride];
            if (ls == -INFINITY) continue;                     // no visible key in this range
            const float w = expf(ls - m);
            den += w;
            float x[PER];
            load_f<PER>(po + s * split_stride * D, x);
#pragma unroll
            for (int i = 0; i < PER; ++i) acc[i] = fmaf(w, x[i], acc[i]);
        }
    }
    const float inv = den > 0.f ? p.out_scale / den : 0.f;
#pragma unroll
    for (int i = 0; i < PER; ++i) acc[i] *= inv;
    store_o<PER>(p.o, (row * p.H + h) * D + lane * PER, p.odtype, acc);
    if (p.lse && lane == 0) {
        const int64_t li = p.varlen ? (int64_t)h * p.total_length + row
                                    : ((row / p.Sq) * p.H + h) * p.Sq + row % p.Sq;
        p.lse[li] = den > 0.f ? m + logf(den) : -INFINITY;
    }
}

int64_t part_rows_of(int B, int Sq, int64_t total_length) {
    return total_length > 0 ? total_length : (int64_t)B * Sq;
}

size_t lse_bytes(int H, int num_splits, int64_t rows) {
    const size_t b = (size_t)num_splits * (size_t)rows * (size_t)H * sizeof(float);
    return (b + 255) & ~(size_t)255;
}

}  // namespace

int launch_combine(const Params &p, cudaStream_t stream) {
    const int64_t items = p.part_rows * p.H;                  // upper bound (varlen: total rows)
    const int64_t blocks = (items + kCombineWarps - 1) / kCombineWarps;
    if (blocks <= 0) return FMHA_OK;
    if (blocks > 0x7fffffff) return FMHA_ERR_UNSUPPORTED;
    void (*kern)(Params) = p.D == 32 ? combine_kernel<32> : p.D == 64 ? combine_kernel<64>
                         : p.D == 128 ? combine_kernel<128> : nullptr;
    if (!kern) return FMHA_ERR_INVALID_ARG;
    // a programmatic dependent of the attention kernel launched just before
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(kCombineWarps * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p) == cudaSuccess ? FMHA_OK : FMHA_ERR_CUDA;
}

}  // namespace fmha

extern "C" {

size_t fmha_fwd_splitkv_workspace_size(int B, int H, int Sq, int D, int num_splits, int64_t total_length) {
    if (B < 0 || H <= 0 || Sq < 0 || (D != 32 && D != 64 && D != 128) || num_splits < 1 ||
        num_splits > fmha::kMaxSplits || total_length < 0)
        return 0;
    const int64_t rows = fmha::part_rows_of(B, Sq, total_length);
    return fmha::lse_bytes(H, num_splits, rows) + (size_t)num_splits * (size_t)rows * H * D * sizeof(float);
}

int fmha_fwd_splitkv(fmha_tensor q, fmha_tensor k, fmha_tensor v, fmha_tensor o, float *lse,
                     int B, int H, int H_k, int Sq, int Sk, int D, float scale, float out_scale,
                     int mask, int causal_type, const int *cu_seqlens_q, const int *cu_seqlens_k,
                     int max_len, int64_t total_length, int num_splits, void *workspace,
                     size_t workspace_bytes, cudaStream_t stream) {
    if (num_splits < 1 || num_splits > fmha::kMaxSplits) return FMHA_ERR_INVALID_ARG;
    fmha::Params p{};
    int rc = fmha::make_params(p, q, k, v, o, lse, B, H, H_k, Sq, Sk, D, scale, out_scale, mask,
                               causal_type, cu_seqlens_q, cu_seqlens_k, max_len, total_length);
    if (rc == 1) return FMHA_OK;
    if (rc != FMHA_OK) return rc;
    const int64_t rows = fmha::part_rows_of(B, p.varlen ? 0 : Sq, p.varlen ? total_length : 0);
    const size_t need = fmha_fwd_splitkv_workspace_size(B, H, p.varlen ? 0 : Sq, D, num_splits,
                                                        p.varlen ? total_length : 0);
    if (!workspace || workspace_bytes < need) return FMHA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(workspace) & 255) return FMHA_ERR_INVALID_ARG;
    // work items (units x splits) are numbered in 32-bit integers on the device
    const int64_t units = p.varlen ? (int64_t)H * (B + total_length / 256 + 1)
                                   : (int64_t)B * H * ((Sq + 255) / 256);
    if (units * num_splits >= (int64_t(1) << 31)) return FMHA_ERR_UNSUPPORTED;
    if ((rc = fmha::check_device()) != FMHA_OK) return rc;
    p.num_splits = num_splits;
    p.part_rows = rows;
    p.part_lse = reinterpret_cast<float *>(workspace);
    p.part_o = reinterpret_cast<float *>(reinterpret_cast<char *>(workspace) +
                                         fmha::lse_bytes(H, num_splits, rows));
    if ((rc = fmha::launch_sm103(p, stream)) != FMHA_OK) return rc;
    return fmha::launch_combine(p, stream);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Split-KV without any allocation
// ---------------------------------------------------------------------------
//
// Some callers cannot allocate device memory at the time they run attention:
// a serving process that reserves all of its HBM once at start-up and treats
// any later cudaMalloc as an error (it can fail, fragment the reservation, or
// stall the device while it synchronises), or a plug-in hosted by a framework
// that owns every device allocation.  For them the scratch of the split-KV
// path lives in this file-scope array instead of a caller workspace.  Every
// GPU that loads the library keeps these bytes reserved until the process
// exits.

namespace fmha {
namespace {

constexpr size_t kNoAllocScratchBytes = FMHA_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch in the current context.  In host code
// the array's name stands for a host-side shadow, not for device memory, so
// the address must come from cudaGetSymbolAddress, with the device current.
// It is looked up on every call rather than cached: the array moves when the
// device's context is destroyed and created again (cudaDeviceReset), and a
// cached address would then point at unmapped memory.
int noalloc_scratch(void **out) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) {
        cudaGetLastError();
        return FMHA_ERR_CUDA;
    }
    *out = ptr;
    return FMHA_OK;
}

}  // namespace
}  // namespace fmha

extern "C" int fmha_fwd_splitkv_noalloc(fmha_tensor q, fmha_tensor k, fmha_tensor v, fmha_tensor o,
                                        float *lse, int B, int H, int H_k, int Sq, int Sk, int D,
                                        float scale, float out_scale, int mask, int causal_type,
                                        const int *cu_seqlens_q, const int *cu_seqlens_k, int max_len,
                                        int64_t total_length, int num_splits, cudaStream_t stream) {
    // the same checks, in the same order, as fmha_fwd_splitkv: an empty problem
    // succeeds and a bad argument gets its own status before the size test
    if (num_splits < 1 || num_splits > fmha::kMaxSplits) return FMHA_ERR_INVALID_ARG;
    fmha::Params p{};
    int rc = fmha::make_params(p, q, k, v, o, lse, B, H, H_k, Sq, Sk, D, scale, out_scale, mask,
                               causal_type, cu_seqlens_q, cu_seqlens_k, max_len, total_length);
    if (rc == 1) return FMHA_OK;
    if (rc != FMHA_OK) return rc;
    const size_t need = fmha_fwd_splitkv_workspace_size(B, H, p.varlen ? 0 : Sq, D, num_splits,
                                                        p.varlen ? total_length : 0);
    if (need == 0) return FMHA_ERR_INVALID_ARG;
    if (need > fmha::kNoAllocScratchBytes) return FMHA_ERR_UNSUPPORTED;   // too big for the array
    void *scratch = nullptr;
    if ((rc = fmha::noalloc_scratch(&scratch)) != FMHA_OK) return rc;
    return fmha_fwd_splitkv(q, k, v, o, lse, B, H, H_k, Sq, Sk, D, scale, out_scale, mask, causal_type,
                            cu_seqlens_q, cu_seqlens_k, max_len, total_length, num_splits, scratch,
                            fmha::kNoAllocScratchBytes, stream);
}
