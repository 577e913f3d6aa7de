// fmha_api.cu -- the C ABI: argument validation and dispatch.
//
// Every argument is checked here, on the host, before anything is launched;
// the kernels assume validated parameters.
#include <cuda_runtime.h>
#include <math.h>
#include <mutex>

#include "fmha_common.h"

namespace fmha {
int gen_read_status(int reset);   // fmha_gen.cu: the generation kernels' status word
int gen_set_wait_limit(unsigned long long ns);   // fmha_gen.cu: its wait limit (0: 4 s)
int gen_set_test_gate(int on);                   // fmha_gen.cu: its producer test gate
int bwd_read_status(int reset);   // fmha_bwd.cu: the backward kernels' status word
int bwd_set_wait_limit(unsigned long long ns);   // fmha_bwd.cu: its wait limit (0: 4 s)
int bwd_set_test_gate(int on);                   // fmha_bwd.cu: its producer test gate
}

namespace fmha {
namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

// Is the current device an sm_103 part?  Cached per device ordinal.
int check_device() {
    static std::mutex mu;
    static int cached[64];            // 0 unknown, 1 ok, 2 unsupported
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return FMHA_ERR_CUDA; }
    if (dev < 0 || dev >= 64) return FMHA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(mu);
    if (cached[dev] == 0) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
            cudaGetLastError();
            return FMHA_ERR_CUDA;
        }
        cached[dev] = (major == 10 && minor == 3) ? 1 : 2;
    }
    return cached[dev] == 1 ? FMHA_OK : FMHA_ERR_UNSUPPORTED;
}

// Validate and fill Params.  Returns FMHA_OK, an error, or 1 for "nothing to do".
int make_params(Params &p, fmha_tensor q, fmha_tensor k, fmha_tensor v, fmha_tensor o,
                float *lse, int B, int H, int H_k, int Sq, int Sk, int D, float scale,
                float out_scale, int mask, int causal_type, const int *cu_q, const int *cu_k,
                int max_len, int64_t total_length) {
    if (B < 0 || H <= 0 || H_k <= 0 || H % H_k != 0) return FMHA_ERR_INVALID_ARG;
    if (D != 32 && D != 64 && D != 128) return FMHA_ERR_INVALID_ARG;
    if (mask < FMHA_MASK_NONE || mask > FMHA_MASK_CAUSAL) return FMHA_ERR_INVALID_ARG;
    if (causal_type != FMHA_CAUSAL_QBEGIN && causal_type != FMHA_CAUSAL_QEND)
        return FMHA_ERR_INVALID_ARG;
    // scale > 0: the kernels take the row max of raw scores before scaling
    if (!isfinite(scale) || !(scale > 0.f) || !isfinite(out_scale)) return FMHA_ERR_INVALID_ARG;
    if ((cu_q == nullptr) != (cu_k == nullptr)) return FMHA_ERR_INVALID_ARG;
    const bool varlen = cu_q != nullptr;
    if (varlen) {
        if (total_length < 0 || max_len < 0) return FMHA_ERR_INVALID_ARG;
        if (total_length > 0 && max_len == 0) return FMHA_ERR_INVALID_ARG;
        if (total_length >= (int64_t(1) << 31)) return FMHA_ERR_UNSUPPORTED;
    } else {
        if (Sq < 0 || Sk < 0) return FMHA_ERR_INVALID_ARG;
    }
    for (int dt : {q.dtype, k.dtype, v.dtype, o.dtype})
        if (dt < FMHA_F16 || dt > FMHA_E4M3) return FMHA_ERR_INVALID_ARG;
    if (k.dtype != q.dtype || v.dtype != q.dtype) return FMHA_ERR_UNSUPPORTED;
    if (o.dtype != q.dtype) return FMHA_ERR_UNSUPPORTED;

    const bool empty = varlen ? (B == 0 || total_length == 0) : (B == 0 || Sq == 0);
    if (empty) return 1;
    if (!q.data || !k.data || !v.data || !o.data) return FMHA_ERR_INVALID_ARG;
    if (!aligned16(q.data) || !aligned16(k.data) || !aligned16(v.data) || !aligned16(o.data))
        return FMHA_ERR_UNSUPPORTED;
    if (lse && (reinterpret_cast<uintptr_t>(lse) & 3)) return FMHA_ERR_INVALID_ARG;
    // coordinates and row indices are kept in 32-bit registers on the device
    if (!varlen && ((int64_t)B * Sq >= (int64_t(1) << 31) || (int64_t)B * Sk >= (int64_t(1) << 31)))
        return FMHA_ERR_UNSUPPORTED;

    p.q = q.data; p.k = k.data; p.v = v.data; p.o = o.data; p.lse = lse;
    p.B = B; p.H = H; p.H_k = H_k; p.D = D; p.group = H / H_k;
    p.Sq = varlen ? 0 : Sq;
    p.Sk = varlen ? 0 : Sk;
    p.scale = scale; p.out_scale = out_scale;
    p.mask = mask; p.causal_type = causal_type;
    p.cu_q = cu_q; p.cu_k = cu_k; p.max_len = max_len;
    p.total_length = varlen ? total_length : 0;
    p.varlen = varlen ? 1 : 0;
    p.dtype = q.dtype; p.odtype = o.dtype;
    p.num_splits = 1;
    p.part_o = nullptr; p.part_lse = nullptr; p.part_rows = 0;
    // up to 128 query rows fill only one of a unit's two Q tiles: pair two
    // query heads of one kv head instead (they share the K/V stream)
    p.hpair = (!varlen && Sq <= 128 && p.group % 2 == 0) ? 1 : 0;
    return FMHA_OK;
}

}  // namespace fmha

extern "C" {

int fmha_fwd(fmha_tensor q, fmha_tensor k, fmha_tensor v, fmha_tensor o, float *lse,
             int B, int H, int H_k, int Sq, int Sk, int D, float scale, float out_scale,
             int mask, int causal_type, const int *cu_seqlens_q, const int *cu_seqlens_k,
             int max_len, int64_t total_length, cudaStream_t stream) {
    fmha::Params p{};
    int rc = fmha::make_params(p, q, k, v, o, lse, B, H, H_k, Sq, Sk, D, scale, out_scale, mask,
                               causal_type, cu_seqlens_q, cu_seqlens_k, max_len, total_length);
    if (rc == 1) return FMHA_OK;
    if (rc != FMHA_OK) return rc;
    if ((rc = fmha::check_device()) != FMHA_OK) return rc;
    return fmha::launch_sm103(p, stream);
}

int fmha_fwd_simt(fmha_tensor q, fmha_tensor k, fmha_tensor v, fmha_tensor o, float *lse,
                  int B, int H, int H_k, int Sq, int Sk, int D, float scale, float out_scale,
                  int mask, int causal_type, const int *cu_seqlens_q, const int *cu_seqlens_k,
                  int max_len, int64_t total_length, cudaStream_t stream) {
    fmha::Params p{};
    int rc = fmha::make_params(p, q, k, v, o, lse, B, H, H_k, Sq, Sk, D, scale, out_scale, mask,
                               causal_type, cu_seqlens_q, cu_seqlens_k, max_len, total_length);
    if (rc == 1) return FMHA_OK;
    if (rc != FMHA_OK) return rc;
    if ((rc = fmha::check_device()) != FMHA_OK) return rc;
    return fmha::launch_simt(p, stream);
}

const char *fmha_status_string(int status) {
    switch (status) {
    case FMHA_OK: return "ok";
    case FMHA_ERR_INVALID_ARG: return "invalid argument";
    case FMHA_ERR_UNSUPPORTED: return "unsupported (dtype combination, alignment or device)";
    case FMHA_ERR_CUDA: return "CUDA runtime or driver error";
    case FMHA_ERR_TIMEOUT: return "a bounded on-device wait expired";
    default: return "unknown status";
    }
}

int fmha_set_wait_limit_ns(unsigned long long ns) {
    const int a = fmha::sm103_set_wait_limit(ns);
    const int b = fmha::gen_set_wait_limit(ns);
    const int c = fmha::bwd_set_wait_limit(ns);
    return a != FMHA_OK ? a : b != FMHA_OK ? b : c;
}

int fmha_set_test_gate(int on) {
    const int a = fmha::sm103_set_test_gate(on);
    const int b = fmha::gen_set_test_gate(on);
    const int c = fmha::bwd_set_test_gate(on);
    return a != FMHA_OK ? a : b != FMHA_OK ? b : c;
}

int fmha_device_status(int reset) {
    const int a = fmha::sm103_read_status(reset);
    const int b = fmha::gen_read_status(reset);
    const int c = fmha::bwd_read_status(reset);
    return a != FMHA_OK ? a : (b != FMHA_OK ? b : c);
}

int fmha_kv_tile_range(int q_row0, int q_rows, int Sq, int Sk, int mask, int causal_type,
                       int tile_n, int *n_tiles, int *n_unmasked) {
    if (!n_tiles || !n_unmasked || tile_n <= 0 || q_row0 < 0 || q_rows < 0 || Sq < 0 || Sk < 0)
        return FMHA_ERR_INVALID_ARG;
    if (mask < FMHA_MASK_NONE || mask > FMHA_MASK_CAUSAL) return FMHA_ERR_INVALID_ARG;
    if (causal_type != FMHA_CAUSAL_QBEGIN && causal_type != FMHA_CAUSAL_QEND)
        return FMHA_ERR_INVALID_ARG;
    fmha::kv_tile_range(q_row0, q_rows, Sq, Sk, mask, causal_type, tile_n, n_tiles, n_unmasked);
    return FMHA_OK;
}

}  // extern "C"
