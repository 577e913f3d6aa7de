// fmha_common.h -- definitions shared by the host launcher and the kernels.
#pragma once

#include <stdint.h>
#include "../../include/fmha.h"

#if defined(__CUDACC__)
#define FMHA_HD __host__ __device__ __forceinline__
#else
#define FMHA_HD inline
#endif

namespace fmha {

// Everything a kernel needs to know about one call, validated on the host.
struct Params {
    const void *q, *k, *v;
    void *o;
    float *lse;
    int B, H, H_k, Sq, Sk, D;
    int group;              // H / H_k
    // head pairs (fixed length, Sq <= 128, H / H_k even): a work unit's two
    // Q tiles are query heads 2i and 2i + 1 (one kv head) over rows [0, Sq),
    // instead of rows [0, 128) and [128, 256) of one head
    int hpair;
    float scale, out_scale;
    int mask, causal_type;
    const int *cu_q, *cu_k; // device, varlen only
    int max_len;
    int64_t total_length;
    int varlen;
    int dtype, odtype;
    // split-KV mode (num_splits > 1 or part_o set): each work unit's key
    // tiles are cut into num_splits contiguous ranges whose normalised fp32
    // partial O [num_splits][part_rows][H][D] and LSE [num_splits][part_rows][H]
    // go to part_o / part_lse instead of o / lse.
    int num_splits;
    float *part_o, *part_lse;
    int64_t part_rows;
};

FMHA_HD int imin(int a, int b) { return a < b ? a : b; }
FMHA_HD int imax(int a, int b) { return a > b ? a : b; }

// Key-tile bounds of one query tile ("CUTLASS Blackwell FMHA 示例完全解析",
// §融合扩展点: the mask classes report a trip count and split it into tiles
// that need the mask and tiles that do not).
//
// Query rows [row0, row0 + rows) of a sequence with sq queries and sk keys.
// Key j is visible to query i iff j < sk and, for a causal mask,
// j <= i + off with off = sk - sq for q-end alignment and 0 for q-begin.
//   n_tiles:    key tiles [0, n_tiles) hold every key visible to some row;
//   n_unmasked: key tiles [0, n_unmasked) are visible to every row in full.
FMHA_HD void kv_tile_range(int row0, int rows, int sq, int sk, int mask, int causal_type,
                           int tile_n, int *n_tiles, int *n_unmasked) {
    const int last_row = imin(row0 + rows, sq) - 1;
    if (last_row < row0 || sk <= 0) { *n_tiles = 0; *n_unmasked = 0; return; }
    const int all_tiles = (sk + tile_n - 1) / tile_n;
    const int full_tiles = sk / tile_n;
    if (mask != FMHA_MASK_CAUSAL) { *n_tiles = all_tiles; *n_unmasked = full_tiles; return; }
    const int off = causal_type == FMHA_CAUSAL_QEND ? sk - sq : 0;
    const int max_key = last_row + off;          // last row sees keys <= max_key
    if (max_key < 0) { *n_tiles = 0; *n_unmasked = 0; return; }
    const int nt = imin(all_tiles, max_key / tile_n + 1);
    const int first_vis = row0 + off + 1;        // first row sees keys < first_vis
    int nu = first_vis > 0 ? first_vis / tile_n : 0;
    nu = imin(imin(nu, full_tiles), nt);
    *n_tiles = nt;
    *n_unmasked = nu;
}

// Argument validation shared by the entry points (fmha_api.cu).  Returns
// FMHA_OK, an error status, or 1 when there is nothing to compute.
int make_params(Params &p, fmha_tensor q, fmha_tensor k, fmha_tensor v, fmha_tensor o, float *lse,
                int B, int H, int H_k, int Sq, int Sk, int D, float scale, float out_scale, int mask,
                int causal_type, const int *cu_q, const int *cu_k, int max_len, int64_t total_length);
int check_device();

// Launchers.  They assume validated parameters.
int launch_simt(const Params &p, cudaStream_t stream);
int launch_sm103(const Params &p, cudaStream_t stream);
int launch_combine(const Params &p, cudaStream_t stream);
int sm103_read_status(int reset);
int sm103_set_wait_limit(unsigned long long ns);   // 0: the default (4 s)
int sm103_set_test_gate(int on);

}  // namespace fmha
