// fmha_simt.cu -- the attention forward on CUDA cores (fp32), a slow
// cross-check of the tensor-core kernel.
//
// One CTA of 128 threads owns 64 query rows of one (batch, head); two threads
// share a row.  Key/value tiles of 64 rows are staged in shared memory as
// fp32.  The softmax is the online form of "fmha sm120 : 超越
// torch.sdpa(flash-attention-2)", §1-§2: running max m and running sum l per
// row, O rescaled by exp(m_old - m_new) when the max grows; the two threads
// of a row combine their partial max and sum with one shuffle.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <math.h>

#include "fmha_common.h"

namespace fmha {
namespace {

constexpr int kRows = 64;     // query rows per CTA
constexpr int kKeys = 64;     // keys per shared-memory tile
constexpr int kThreads = 128;

__device__ __forceinline__ float load_elem(const void *base, int64_t idx, int dtype) {
    if (dtype == FMHA_BF16) {
        return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(base)[idx]);
    } else if (dtype == FMHA_F16) {
        return __half2float(reinterpret_cast<const __half *>(base)[idx]);
    } else {
        __nv_fp8_storage_t b = reinterpret_cast<const __nv_fp8_storage_t *>(base)[idx];
        return __half2float(__half(__nv_cvt_fp8_to_halfraw(b, __NV_E4M3)));
    }
}

__device__ __forceinline__ void store_elem(void *base, int64_t idx, int dtype, float x) {
    if (dtype == FMHA_BF16) {
        reinterpret_cast<__nv_bfloat16 *>(base)[idx] = __float2bfloat16_rn(x);
    } else if (dtype == FMHA_F16) {
        reinterpret_cast<__half *>(base)[idx] = __float2half_rn(x);
    } else {
        reinterpret_cast<__nv_fp8_storage_t *>(base)[idx] =
            __nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
    }
}

template <int D>
__global__ void __launch_bounds__(kThreads) simt_kernel(const Params p) {
    extern __shared__ float smem[];
    float *Qs = smem;                            // [kRows][D]
    float *Ks = Qs + kRows * D;                  // [kKeys][D + 1]
    float *Vs = Ks + kKeys * (D + 1);            // [kKeys][D]
    float *Ps = Vs + kKeys * D;                  // [kRows][kKeys + 1]

    const int b = blockIdx.z, h = blockIdx.y;
    const int row0 = blockIdx.x * kRows;
    int64_t q_start, k_start;
    int sq, sk;
    if (p.varlen) {
        q_start = p.cu_q[b]; sq = p.cu_q[b + 1] - p.cu_q[b];
        k_start = p.cu_k[b]; sk = p.cu_k[b + 1] - p.cu_k[b];
    } else {
        q_start = (int64_t)b * p.Sq; sq = p.Sq;
        k_start = (int64_t)b * p.Sk; sk = p.Sk;
    }
    if (row0 >= sq) return;
    const int g = h / p.group;
    const int t = threadIdx.x;
    const int r = t >> 1, half = t & 1;
    const int i = row0 + r;                      // this thread's query row
    const int off = (p.mask == FMHA_MASK_CAUSAL && p.causal_type == FMHA_CAUSAL_QEND) ? sk - sq : 0;
    const bool causal = p.mask == FMHA_MASK_CAUSAL;

    for (int idx = t; idx < kRows * D; idx += kThreads) {
        const int rr = idx / D, d = idx % D;
        const int ii = row0 + rr;
        Qs[idx] = ii < sq ? load_elem(p.q, ((q_start + ii) * p.H + h) * (int64_t)D + d, p.dtype) : 0.f;
    }
    int n_tiles, n_unmasked;
    kv_tile_range(row0, kRows, sq, sk, p.mask, p.causal_type, kKeys, &n_tiles, &n_unmasked);

    constexpr int DH = D / 2;                    // output columns per thread
    float acc[DH];
#pragma unroll
    for (int d = 0; d < DH; ++d) acc[d] = 0.f;
    float m = -INFINITY, l = 0.f;

    for (int j = 0; j < n_tiles; ++j) {
        __syncthreads();
        const int k0 = j * kKeys;
        for (int idx = t; idx < kKeys * D; idx += kThreads) {
            const int kk = idx / D, d = idx % D;
            const int key = k0 + kk;
            float kv = 0.f, vv = 0.f;
            if (key < sk) {
                const int64_t e = ((k_start + key) * p.H_k + g) * (int64_t)D + d;
                kv = load_elem(p.k, e, p.dtype);
                vv = load_elem(p.v, e, p.dtype);
            }
            Ks[kk * (D + 1) + d] = kv;
            Vs[idx] = vv;
        }
        __syncthreads();

        float s[kKeys / 2];
        float mt = -INFINITY;
#pragma unroll 4
        for (int c = 0; c < kKeys / 2; ++c) {
            const int kk = 2 * c + half;
            float dot = 0.f;
#pragma unroll 8
            for (int d = 0; d < D; ++d) dot = fmaf(Qs[r * D + d], Ks[kk * (D + 1) + d], dot);
            const int key = k0 + kk;
            const bool vis = key < sk && (!causal || key <= i + off) && i < sq;
            s[c] = vis ? dot * p.scale : -INFINITY;
            mt = fmaxf(mt, s[c]);
        }
        mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 1));
        const float m_new = fmaxf(m, mt);
        float ls = 0.f;
        if (m_new != -INFINITY) {
            const float alpha = expf(m - m_new);     // m == -inf gives 0
            l *= alpha;
#pragma unroll
            for (int d = 0; d < DH; ++d) acc[d] *= alpha;
#pragma unroll 4
            for (int c = 0; c < kKeys / 2; ++c) {
                const float pv = expf(s[c] - m_new);  // masked: exp(-inf) = 0
                Ps[r * (kKeys + 1) + 2 * c + half] = pv;
                ls += pv;
            }
            m = m_new;
        } else {
#pragma unroll 4
            for (int c = 0; c < kKeys / 2; ++c) Ps[r * (kKeys + 1) + 2 * c + half] = 0.f;
        }
        ls += __shfl_xor_sync(0xffffffffu, ls, 1);
        l += ls;
        __syncwarp();
        for (int kk = 0; kk < kKeys; ++kk) {
            const float pv = Ps[r * (kKeys + 1) + kk];
#pragma unroll
            for (int d = 0; d < DH; ++d) acc[d] = fmaf(pv, Vs[kk * D + half * DH + d], acc[d]);
        }
    }

    if (i < sq) {
        const float inv = l > 0.f ? p.out_scale / l : 0.f;
        const int64_t obase = ((q_start + i) * p.H + h) * (int64_t)D + half * DH;
#pragma unroll
        for (int d = 0; d < DH; ++d) store_elem(p.o, obase + d, p.odtype, acc[d] * inv);
        if (p.lse && half == 0) {
            const int64_t li = p.varlen ? (int64_t)h * p.total_length + q_start + i
                                        : ((int64_t)b * p.H + h) * p.Sq + i;
            p.lse[li] = l > 0.f ? m + logf(l) : -INFINITY;
        }
    }
}

template <int D>
int launch_d(const Params &p, cudaStream_t stream) {
    const size_t smem = sizeof(float) * (kRows * D + kKeys * (D + 1) + kKeys * D + kRows * (kKeys + 1));
    static bool attr_set = false;   // per process; harmless to repeat
    if (!attr_set) {
        if (cudaFuncSetAttribute(simt_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem) != cudaSuccess) {
            cudaGetLastError();
            return FMHA_ERR_CUDA;
        }
        attr_set = true;
    }
    const int rows = p.varlen ? p.max_len : p.Sq;
    if (rows == 0) return FMHA_OK;
    dim3 grid((rows + kRows - 1) / kRows, p.H, p.B);
    simt_kernel<D><<<grid, kThreads, smem, stream>>>(p);
    if (cudaGetLastError() != cudaSuccess) return FMHA_ERR_CUDA;
    return FMHA_OK;
}

}  // namespace

int launch_simt(const Params &p, cudaStream_t stream) {
    switch (p.D) {
    case 32: return launch_d<32>(p, stream);
    case 64: return launch_d<64>(p, stream);
    case 128: return launch_d<128>(p, stream);
    default: return FMHA_ERR_INVALID_ARG;
    }
}

}  // namespace fmha
