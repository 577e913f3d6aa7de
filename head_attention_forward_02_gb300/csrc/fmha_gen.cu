// fmha_gen.cu -- generation-phase attention forward for sm_103a: one new query
// token per sequence against that sequence's entry of a K/V cache, and the
// merge of the per-chunk partial results.
//
// Operation ("CUTLASS Blackwell FMHA 示例完全解析", §FMHA for Blackwell 生成阶段):
// for sequence b, query head h, kv head g = h / G (G = H / H_k query heads per
// kv head), cache entry e = batch_idx ? batch_idx[b] : b and L = seqlen[b]
// cached tokens, the keys are K_cache[e, 0..L-1, g] and, unless the call is
// cache-only, the new token's K_new[b, g], which is also written into the
// cache at row L (V alike); O[b, h] = softmax(scale * q[b, h] K^T) V.  The
// page fixes head dim 128 and one query-head group per thread block.  Element
// types: fp16, bf16 and fp8 e4m3 (kind::f8f6f4 MMAs; the weights P are
// rounded to e4m3 before P.V, their row sum is kept in fp32).
//
// The work is memory bound: every cached K/V byte is read once, and a group of
// G <= 32 query heads does 4 * G flops per cached element pair.  The design
// therefore aims at HBM bandwidth: the key range of every (sequence, kv head)
// is cut into chunks so that all SMs stream at once, each CTA keeps a ring of
// three 64 KB K/V stages in flight through TMA, and the contraction runs on
// the tensor cores with the roles swapped so that the small head group is the
// N dimension: per 128-row tile block,
// S^T = K Q^T (M = 128 keys, N = 32 padded heads, K = 128) and
// O^T += V^T P^T (M = 128 = head dim, N = 32, K = 128 keys); a 16-bit tile is
// one block, an e4m3 tile two (the same 64 KB).  Thread i of the softmax
// warps owns row i of every block (TMEM lane i) and, in the epilogue, head
// dimension i of O^T.  The row maximum is kept lazily per head (rescale only
// when a score exceeds the reference by 2^8), so the common tile needs no
// cross-thread reduction; a named-barrier vote finds the rare tile that does.
// Each chunk writes a normalised fp32 partial O and its LSE; a merge kernel
// combines the chunks of every (b, h) by their LSE weights.
#include <cuda.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "fmha_common.h"

namespace fmha {

__device__ int g_gen_status;   // FMHA_OK, or the first error a generation kernel met
// the bounded waits' limit (ns); set from the host through fmha_set_wait_limit_ns
__device__ unsigned long long g_gen_wait_ns = 4000000000ull;
// test hook (fmha_set_test_gate): when set, the producer first waits for a
// flag that nothing writes, so that bounded wait runs out before any copy
__device__ int g_gen_test_gate;
__device__ int g_gen_test_flag;   // never written

namespace {

constexpr int kD = 128;                 // head dim
constexpr int kKT = 128;                // rows per tile block (MMA M of S^T): keys, or keys x 2 heads
constexpr int kNP = 32;                 // query heads of a group, padded (MMA N)
constexpr int kNSMax = 6;               // K/V ring stages at most (a K and a V tile each)
constexpr int kBarBytes = 2048;         // barrier and scratch block
constexpr int kSoftWarpsMax = 8;        // softmax warps of the widest layout
constexpr int kPanelBytes = kKT * 128;  // 128 rows of one 128-byte swizzled panel
constexpr int kQPanelBytes = kNP * 128;
constexpr int kQSlots = 2;                            // Q tiles of consecutive work items

// Sizes and layouts of one element type: 16-bit (f16, bf16) or e4m3.  A 128-dim
// row is two 128-byte swizzle panels of 64 elements, or one of 128.  A tile
// is BLK blocks of 128 rows; each block has its own S^T columns and P^T
// buffer, and every block's P.V accumulates into the one O^T.  e4m3 tiles
// have two blocks, so that a tile carries as many bytes (64 KB of K and V)
// as a 16-bit one and the per-tile hand-offs cost the same per byte.
template <int ELEM, int BLK_>
struct GenCfg {
    static constexpr bool FP8 = ELEM == FMHA_E4M3;
    static constexpr int BLK = BLK_;                      // 128-row blocks per tile
    static constexpr int E = FP8 ? 1 : 2;                 // bytes per element
    static constexpr int PANELS = kD * E / 128;
    static constexpr int BOX = 128 / E;                   // elements per panel row
    static constexpr int BLK_BYTES = PANELS * kPanelBytes;    // one block: 128 rows x 128 dims
    static constexpr int TILE_BYTES = BLK * BLK_BYTES;        // the K (or V) half of a stage
    static constexpr int Q_BYTES = PANELS * kQPanelBytes;     // 32 heads x 128 dims
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;        // K blocks, then V blocks
    static constexpr int P_ROW = kNP * E;                 // bytes of one key's P^T row (32 heads)
    static constexpr int P_BYTES = kKT * P_ROW;           // P^T of one block
    static constexpr uint64_t P_SWZ = FP8 ? 6 : 4;        // 32-byte or 64-byte swizzle of P^T
    static constexpr int MMA_K = FP8 ? 32 : 16;           // K of one tcgen05.mma
    static constexpr uint32_t FMT = ELEM == FMHA_BF16 ? 1u : 0u;   // kind::f16: f16 0, bf16 1; f8f6f4: e4m3 0
    // TMEM: S^T buffers in [0, SCOLS) and [SCOLS, 2 SCOLS) (block i of a
    // buffer in its columns [32 i, 32 i + 32)), O^T in [2 SCOLS, 2 SCOLS + 32)
    static constexpr int SCOLS = BLK * kNP;
    static constexpr int O_COL = 2 * SCOLS;
    static constexpr uint32_t TMEM_COLS = O_COL + kNP <= 128 ? 128 : 256;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_KV = OFF_Q + kQSlots * Q_BYTES;
    static constexpr int NS = STAGE_BYTES >= 65536 ? 3 : 6;   // K/V ring stages: about 192 KB in flight
    static constexpr int OFF_P = OFF_KV + NS * STAGE_BYTES;
    static constexpr int OFF_BARS = OFF_P + 2 * BLK * P_BYTES;
    static constexpr int SMEM_BYTES = OFF_BARS + kBarBytes + 1024;   // barriers and scratch, 1 KB alignment
    static_assert(SMEM_BYTES <= 227 * 1024 && NS <= kNSMax, "shared memory budget");
    static_assert(O_COL + kNP <= (int)TMEM_COLS, "TMEM budget");
};

// Blocks per tile of an element type and warp layout: two for e4m3, except in
// the eight-warp layout, whose two column groups of 16 already hold 168
// registers a thread with one block
template <int ELEM, int MODE>
struct GenBlk {
    static constexpr int value = ELEM == FMHA_E4M3 && MODE != 2 ? 2 : 1;
};
constexpr unsigned long long kTimeoutNs = 4000000000ull;   // the default wait limit
constexpr unsigned long long kDrainNs = 200000000ull;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.0f;    // rescale when a head's max grows by more than 2^8

struct GenParams {
    const void *q, *k_new, *v_new;      // q [B, H, D]; new K/V [B, H_k, D] (insert mode)
    void *k_cache, *v_cache;            // [B_cache, S_max, H_k, D]
    const int *seqlen, *batch_idx;      // device int32 [B]; batch_idx may be NULL
    void *o;                            // [B, H, D]
    float *lse;                         // [B, H] or NULL
    float *part_o, *part_lse;           // [B*H][max_seg][D], [B*H][max_seg]
    int B, H, H_k, G, B_cache, S_max;
    int GP;                             // kv heads per work unit: 2 (adjacent heads together) or 1
    int TK;                             // keys per tile: 128 x blocks per tile / GP
    int NU;                             // work units per sequence: H_k / GP
    int max_seg;                        // partial results per (sequence, head): tiles of S_max + 1
    int ncta;                           // CTAs of the attention kernel (the stream-K split)
    int insert, dtype;
    float c;                            // scale * log2(e)
    float out_scale;
};

struct GenSched {
    int64_t per, G0, G1;                // this CTA's tiles [G0, G1)
    int64_t off0;                       // first tile of sequence b0
    int b0;                             // first sequence with a tile at or past G0
};

struct GenBars {
    uint64_t q_full[kQSlots], q_empty[kQSlots], o_full, drain;
    uint64_t s_full[2], s_free[2], p_full[2], pv_done[2];   // per S^T / P^T buffer
    uint64_t kv_full[kNSMax], kv_empty[kNSMax];
    uint32_t tmem_base;
    int abort;
    float red[kSoftWarpsMax][kNP];      // per-warp partial max / sum of each column
    float alpha[kNP], mref[kNP];        // rescale factors and reference maxima of every column
    GenSched sched;
};
static_assert(sizeof(GenBars) <= kBarBytes, "barrier block");

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait: the phase completes, the CTA aborts, or g_gen_wait_ns pass (then
// the timeout is recorded and the abort flag raised).
__device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, volatile int *abort_flag) {
    const unsigned long long t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63) == 0) {
            if (*abort_flag) return false;
            if (globaltimer() - t0 > g_gen_wait_ns) {
                *abort_flag = 1;
                atomicExch(&g_gen_status, FMHA_ERR_TIMEOUT);
                return false;
            }
        }
    }
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    return mbar_wait_slow(bar, parity, abort_flag);
}

// Bounded wait that ignores the abort flag (only while draining).
__device__ __noinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity) {
    const unsigned long long t0 = globaltimer();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer() - t0 > kDrainNs) return false;
    }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, uint32_t bar, int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *map, uint32_t bar, int c0, int c1,
                                            int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }


// Shared-memory matrix descriptor: start address and leading / stride byte
// offsets in 16-byte units, descriptor version 1, swizzle mode (128 B = 2,
// 64 B = 4).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint64_t swz) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (swz << 61);
}


// Warp-collective forms: the whole (converged) warp executes them with
// warp-uniform operands and one elected lane issues the instruction.
template <bool FP8>
__device__ __forceinline__ void mma_ss_e(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    if constexpr (FP8) {
        asm volatile(
            "{\n.reg .pred p, e;\nsetp.ne.b32 p, %4, 0;\nelect.sync _|e, 0xffffffff;\n"
            "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
            "l"(a), "l"(b), "r"(idesc), "r"(acc)
            : "memory");
    } else {
        asm volatile(
            "{\n.reg .pred p, e;\nsetp.ne.b32 p, %4, 0;\nelect.sync _|e, 0xffffffff;\n"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
            "l"(a), "l"(b), "r"(idesc), "r"(acc)
            : "memory");
    }
}

__device__ __forceinline__ void tc_commit_e(uint32_t bar) {
    asm volatile(
        "{\n.reg .pred e;\nelect.sync _|e, 0xffffffff;\n"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}\n" ::"r"(bar)
        : "memory");
}

// Bounded wait by a whole warp: true in every lane, or false in every lane.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag) {
    const bool r = mbar_wait(bar, parity, abort_flag);
    return __all_sync(0xffffffffu, r);
}

// Instruction descriptor: fp32 accumulator, A/B format (kind::f16: 0 = f16,
// 1 = bf16; kind::f8f6f4: 0 = e4m3),
// A and B major-ness (0 = K-major, 1 = MN-major), N, M = 128.
__host__ __device__ constexpr uint32_t gen_idesc(uint32_t fmt, bool a_mn, bool b_mn) {
    return (1u << 4) | (fmt << 7) | (fmt << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
           ((uint32_t)(kNP >> 3) << 17) | ((uint32_t)(kKT >> 4) << 24);
}

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// 32 consecutive TMEM columns of this thread's lane (32x32b shape).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

// 32 lanes x N columns for N = 4, 8, 16 (32: tmem_ld32)
template <int N>
__device__ __forceinline__ void tmem_ld_n(uint32_t taddr, uint32_t (&r)[N]) {
    if constexpr (N == 4) {
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                     : "r"(taddr));
    } else if constexpr (N == 8) {
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                     : "r"(taddr));
    } else if constexpr (N == 16) {
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
            "%14, %15}, [%16];"
            : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
              "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
            : "r"(taddr));
    } else {
        static_assert(N == 32, "tcgen05.ld width");
        tmem_ld32(taddr, r);
    }
}

// Wait for this thread's TMEM loads; the register operands tie the values to the wait.
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[32]);
template <int N>
__device__ __forceinline__ void tmem_wait_ld_n(uint32_t (&r)[N]) {
    if constexpr (N == 4) {
        asm volatile("tcgen05.wait::ld.sync.aligned;" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3])::"memory");
    } else if constexpr (N == 8) {
        asm volatile("tcgen05.wait::ld.sync.aligned;"
                     : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7])
                     :
                     : "memory");
    } else if constexpr (N == 16) {
        asm volatile("tcgen05.wait::ld.sync.aligned;"
                     : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                       "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                       "+r"(r[15])
                     :
                     : "memory");
    } else {
        tmem_wait_ld(r);
    }
}

// Wait for this thread's TMEM loads; the register operands tie the values to the wait.
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                   "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                   "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]),
        "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),
        "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

template <int N>
__device__ __forceinline__ void tmem_st_n(uint32_t taddr, const uint32_t (&r)[N]) {
    if constexpr (N == 4) {
        asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(r[0]),
                     "r"(r[1]), "r"(r[2]), "r"(r[3])
                     : "memory");
    } else if constexpr (N == 8) {
        asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
                     "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                     : "memory");
    } else if constexpr (N == 16) {
        asm volatile(
            "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
            "%14, %15, %16};" ::"r"(taddr),
            "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
            "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
            : "memory");
    } else {
        static_assert(N == 32, "tcgen05.st width");
        tmem_st32(taddr, r);
    }
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Named barrier 1 over the N softmax threads, with a vote.
template <int N>
__device__ __forceinline__ void soft_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(N) : "memory");
}
template <int N>
__device__ __forceinline__ bool soft_all(bool v) {
    uint32_t r;
    asm volatile("{\n.reg .pred p, q;\nsetp.ne.u32 p, %1, 0;\nbar.red.and.pred q, 1, %2, p;\nselp.u32 %0, 1, 0, q;\n}\n"
                 : "=r"(r)
                 : "r"((uint32_t)v), "n"(N)
                 : "memory");
    return r != 0;
}
template <int N>
__device__ __forceinline__ bool soft_any(bool v) {
    uint32_t r;
    asm volatile("{\n.reg .pred p, q;\nsetp.ne.u32 p, %1, 0;\nbar.red.or.pred q, 1, %2, p;\nselp.u32 %0, 1, 0, q;\n}\n"
                 : "=r"(r)
                 : "r"((uint32_t)v), "n"(N)
                 : "memory");
    return r != 0;
}

template <bool BF>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    uint32_t r;
    if constexpr (BF) asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    else asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// four values to e4m3 (round to nearest even, saturating), first value in the low byte
__device__ __forceinline__ uint32_t pack4_e4m3(float a, float b, float c, float d) {
    const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
    return lo | (hi << 16);
}

// ---------------------------------------------------------------------------
// Work items: (sequence b, chunk c of its keys, unit u), u fastest.  A unit is
// one kv head, or two adjacent kv heads (GP = 2) whose query groups together
// fill at most the 32 columns of S^T (tile shapes: Unit below).  One key's
// rows of two adjacent heads are contiguous in the cache and the two heads'
// loads of a tile go out back to back, so every K/V row the tile reads is
// twice as long; fetched alone, a 128-byte e4m3 row cost about 1.5x its size
// in DRAM traffic on this part, and a pair of them exactly their size.
// ---------------------------------------------------------------------------

// Keys of sequence b: its cached tokens, plus the new one unless cache-only.
// A length outside [0, S_max - insert] is clamped and reported.
__device__ __forceinline__ int gen_tokens(const GenParams &p, int b, bool report) {
    int L = p.seqlen[b];
    const int hi = p.S_max - p.insert;
    if (L < 0 || L > hi) {
        if (report) atomicCAS(&g_gen_status, FMHA_OK, FMHA_ERR_INVALID_ARG);
        L = L < 0 ? 0 : hi;
    }
    return L;
}

__device__ __forceinline__ int gen_entry(const GenParams &p, int b, bool report) {
    int e = p.batch_idx ? p.batch_idx[b] : b;
    if (e < 0 || e >= p.B_cache) {
        if (report) atomicCAS(&g_gen_status, FMHA_OK, FMHA_ERR_INVALID_ARG);
        e = -1;   // reads of a missing entry are zero-filled; no insert
    }
    return e;
}

// Shape of a work unit (kv heads) and of its tiles (keys per tile, and which
// kv head and key row r of block i holds).  One block: a one-head tile is 128
// keys; a two-head tile is 64 keys x 2 heads, rows 0-63 the first head and
// 64-127 the second.  Two blocks: a one-head tile is 256 keys, block i keys
// [128 i, 128 i + 128); a two-head tile is 128 keys, block i the head g + i.
template <bool TWO_, int BLK_>
struct Unit {
    static constexpr bool TWO = TWO_;
    static constexpr int BLK = BLK_;
    static constexpr int GP = TWO ? 2 : 1;
    static constexpr int TK = kKT * BLK / GP;
    static __device__ __forceinline__ int row_head(int i, int r) { return BLK == 2 ? (TWO ? i : 0) : (TWO ? r >> 6 : 0); }
    static __device__ __forceinline__ int row_key(int i, int r) { return BLK == 2 ? (TWO ? r : kKT * i + r) : (TWO ? r & 63 : r); }
};

// Warp layout of a kernel instantiation.
//   MODE 0: one kv head per unit; 4 softmax warps, one column group
//   MODE 1: two kv heads per unit; 4 softmax warps (one-block tiles: a column
//           group of two warps per head; two-block tiles: every warp takes
//           both heads, one per block)
//   MODE 2: one kv head per unit; 8 softmax warps, two column groups of 16
//           (query groups wider than 16: the exponentials of a tile are
//           shared by twice the threads)
// The producer and MMA warps follow the softmax warps.
template <int MODE>
struct Layout {
    static constexpr bool TWO = MODE == 1;
    static constexpr int SW = MODE == 2 ? 8 : 4;
    static constexpr int PROD = SW, MMA = SW + 1;
    static constexpr int THREADS = (SW + 2) * 32;
};

// Tiles of tk keys covering sequence b's keys
__device__ __forceinline__ int gen_tiles(const GenParams &p, int b, int tk) {
    return (gen_tokens(p, b, false) + p.insert + tk - 1) / tk;
}

// Stream-K split: the tiles of every (sequence b, unit u) pair, in (b, u)
// order, form one sequence of T tiles; CTA i takes tiles
// [i * per, (i + 1) * per) with per = ceil(T / gridDim.x), so every CTA
// streams the same amount of K/V whatever the lengths.  A CTA's range is cut
// at pair boundaries into segments; segment s of a pair is its part in the
// s-th CTA that covers the pair, and writes partial slot s.

// One warp: T, this CTA's range, and where its first segment starts.
template <class U>
__device__ void gen_schedule(const GenParams &p, GenSched *sc, int lane) {
    int64_t T = 0;
    for (int b = lane; b < p.B; b += 32) T += (int64_t)p.NU * gen_tiles(p, b, U::TK);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) T += __shfl_xor_sync(0xffffffffu, T, o);
    const int64_t per = (T + gridDim.x - 1) / gridDim.x;
    const int64_t G0 = min((int64_t)blockIdx.x * per, T), G1 = min(G0 + per, T);
    int b0 = p.B;
    int64_t off0 = T, base = 0;
    for (int bb = 0; bb < p.B && G0 < G1; bb += 32) {
        const int b = bb + lane;
        const int64_t n = b < p.B ? (int64_t)p.NU * gen_tiles(p, b, U::TK) : 0;
        int64_t incl = n;                 // inclusive prefix over the 32 sequences
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        const unsigned hit = __ballot_sync(0xffffffffu, n > 0 && base + incl > G0);
        if (hit) {
            const int l = __ffs(hit) - 1;
            b0 = bb + l;
            off0 = __shfl_sync(0xffffffffu, base + incl - n, l);
            break;
        }
        base += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
        sc->per = per;
        sc->G0 = G0;
        sc->G1 = G1;
        sc->b0 = b0;
        sc->off0 = off0;
    }
}

struct GenItem {
    int b, g, entry, L, k0, k1;         // keys [k0, k1) of sequence b, kv heads g .. g + GP - 1
    int seg;                            // partial slot of this segment
    bool len_ok;                        // seqlen[b] was within [0, S_max - insert]
};

struct GenCursor {                      // next pair (b, unit u) and its first tile
    int b = -1, u = 0;
    int64_t off = 0;
};

template <class U>
__device__ bool gen_next(const GenParams &p, const GenSched &sc, GenCursor &cur, GenItem &it, bool report) {
    if (cur.b < 0) {
        cur.b = sc.b0;
        cur.u = 0;
        cur.off = sc.off0;
    }
    for (;;) {
        if (cur.b >= p.B || cur.off >= sc.G1) return false;
        const int nt = gen_tiles(p, cur.b, U::TK);
        const int64_t end = cur.off + nt;
        const bool hit = nt > 0 && end > sc.G0;
        if (hit) {
            const int64_t t0 = max(sc.G0, cur.off) - cur.off, t1 = min(sc.G1, end) - cur.off;
            const bool first = t0 == 0 && cur.u == 0;      // reports once per sequence
            it.b = cur.b;
            it.g = cur.u * U::GP;
            it.L = gen_tokens(p, cur.b, report && first);
            it.len_ok = p.seqlen[cur.b] == it.L;
            it.entry = gen_entry(p, cur.b, report && first);
            it.k0 = (int)(t0 * U::TK);
            it.k1 = imin((int)(t1 * U::TK), it.L + p.insert);
            it.seg = (int)(blockIdx.x - cur.off / sc.per);
        }
        cur.off = end;
        if (++cur.u == p.NU) {
            cur.u = 0;
            ++cur.b;
        }
        if (hit) return true;
    }
}

// ---------------------------------------------------------------------------
// Roles
// ---------------------------------------------------------------------------

// TMA producer: per item, the new token's row into the cache (when this chunk
// holds it), the 32-head Q tile, then the chunk's K/V tiles into the ring.
template <class C, class U>
__device__ void gen_producer(const GenParams &p, const GenSched &sc, const CUtensorMap *tmQ,
                             const CUtensorMap *tmK, const CUtensorMap *tmV, uint8_t *smem, GenBars *bars) {
    constexpr bool TWO = U::TWO;
    volatile int *abort_flag = &bars->abort;
    prefetch_tmap(tmQ);
    prefetch_tmap(tmK);
    prefetch_tmap(tmV);
    uint32_t fill = 0, qn = 0;
    bool ok = true;
    if (g_gen_test_gate) {
        // a flag nothing sets: the wait runs out, records the timeout and
        // raises the abort flag; no copy has been issued yet
        const volatile int *flag = &g_gen_test_flag;
        const unsigned long long t0 = globaltimer();
        for (uint32_t it = 1; !*flag; ++it) {
            if ((it & 63) == 0 && (*abort_flag || globaltimer() - t0 > g_gen_wait_ns)) {
                *abort_flag = 1;
                atomicExch(&g_gen_status, FMHA_ERR_TIMEOUT);
                break;
            }
        }
        ok = false;
    }
    GenCursor cur;
    while (ok) {
        GenItem it;
        if (!gen_next<U>(p, sc, cur, it, true)) break;
        if (p.insert && it.len_ok && it.entry >= 0 && it.L >= it.k0 && it.L < it.k1) {
            // K and V rows of the new token (128 elements per kv head of the
            // unit, contiguous); the async proxy (TMA) reads row L below, so
            // order these generic writes before it
            const int64_t src = ((int64_t)it.b * p.H_k + it.g) * kD * C::E;
            const int64_t dst = (((int64_t)it.entry * p.S_max + it.L) * p.H_k + it.g) * kD * C::E;
            const uint4 *kn = reinterpret_cast<const uint4 *>(static_cast<const uint8_t *>(p.k_new) + src);
            const uint4 *vn = reinterpret_cast<const uint4 *>(static_cast<const uint8_t *>(p.v_new) + src);
            uint4 *kc = reinterpret_cast<uint4 *>(static_cast<uint8_t *>(p.k_cache) + dst);
            uint4 *vc = reinterpret_cast<uint4 *>(static_cast<uint8_t *>(p.v_cache) + dst);
#pragma unroll 4
            for (int i = 0; i < U::GP * kD * C::E / 16; ++i) {
                kc[i] = kn[i];
                vc[i] = vn[i];
            }
            asm volatile("fence.proxy.async.global;" ::: "memory");
        }
        // Q slot qn % 2: free once the S^T MMAs of the item two back are done,
        // so the K/V ring keeps streaming across item boundaries
        const int qs = qn % kQSlots;
        const uint32_t qr = qn / kQSlots;
        if (qr > 0 && !mbar_wait(smem_u32(&bars->q_empty[qs]), (qr - 1) & 1, abort_flag)) {
            ok = false;
            break;
        }
        const uint32_t qb = smem_u32(&bars->q_full[qs]);
        mbar_expect_tx(qb, C::Q_BYTES);
        // 32 query heads from the unit's first; a two-head unit takes two
        // 16-row halves, the second from the second kv head's first query
        const int qrow = it.b * p.H + it.g * p.G;
        const uint32_t qdst = smem_u32(smem + C::OFF_Q + qs * C::Q_BYTES);
#pragma unroll
        for (int pn = 0; pn < C::PANELS; ++pn) {
            tma_load_2d(qdst + pn * kQPanelBytes, tmQ, qb, pn * C::BOX, qrow);
            if (TWO) tma_load_2d(qdst + pn * kQPanelBytes + kQPanelBytes / 2, tmQ, qb, pn * C::BOX, qrow + p.G);
        }
        ++qn;
        for (int k = it.k0; k < it.k1; k += U::TK) {
            const int st = fill % C::NS;
            const uint32_t rnd = fill / C::NS;
            if (rnd > 0 && !mbar_wait(smem_u32(&bars->kv_empty[st]), (rnd - 1) & 1, abort_flag)) {
                ok = false;
                break;
            }
            const uint32_t fb = smem_u32(&bars->kv_full[st]);
            mbar_expect_tx(fb, C::STAGE_BYTES);
            const uint32_t dst = smem_u32(smem + C::OFF_KV + st * C::STAGE_BYTES);
            const int e = it.entry >= 0 ? it.entry : p.B_cache;   // out of range: zero fill
            // one box per block, or, in a one-block two-head tile, one per
            // head (rows [64 h2, 64 h2 + 64) are head g + h2); the heads' loads
            // go out back to back, so each key's rows of both heads (adjacent
            // in the cache) are fetched together
            constexpr int NBOX = C::BLK == 2 ? 2 : U::GP;
            constexpr int BOX_ROWS = kKT * C::BLK / NBOX;
#pragma unroll
            for (int x = 0; x < NBOX; ++x) {
                // block x of a two-block tile, or rows [64 x, 64 x + 64) of each panel
                const uint32_t ro = (uint32_t)(C::BLK == 2 ? x * C::BLK_BYTES : x * BOX_ROWS * 128);
                const int hx = C::BLK == 2 ? U::row_head(x, 0) : x;
                const int kx = k + (C::BLK == 2 ? U::row_key(x, 0) : 0);
#pragma unroll
                for (int pn = 0; pn < C::PANELS; ++pn) {
                    tma_load_4d(dst + pn * kPanelBytes + ro, tmK, fb, pn * C::BOX, it.g + hx, kx, e);
                    tma_load_4d(dst + C::TILE_BYTES + pn * kPanelBytes + ro, tmV, fb, pn * C::BOX, it.g + hx, kx, e);
                }
            }
            ++fill;
        }
    }
    if (ok) {
        // every stage's and the Q tile's last release must arrive before exit
        for (int st = 0; st < C::NS; ++st) {
            const uint32_t nf = fill > (uint32_t)st ? (fill - st + C::NS - 1) / C::NS : 0;
            if (nf && !mbar_wait(smem_u32(&bars->kv_empty[st]), (nf - 1) & 1, abort_flag)) break;
        }
        for (uint32_t f = qn > kQSlots ? qn - kQSlots : 0; f < qn; ++f)
            if (!mbar_wait(smem_u32(&bars->q_empty[f % kQSlots]), (f / kQSlots) & 1, abort_flag)) break;
    } else {
        // aborted: let the copies already issued land before the CTA exits
        const uint32_t first = fill > (uint32_t)C::NS ? fill - C::NS : 0;
        for (uint32_t f = first; f < fill; ++f) mbar_wait_drain(smem_u32(&bars->kv_full[f % C::NS]), (f / C::NS) & 1);
        for (uint32_t f = qn > kQSlots ? qn - kQSlots : 0; f < qn; ++f)
            mbar_wait_drain(smem_u32(&bars->q_full[f % kQSlots]), (f / kQSlots) & 1);
    }
}

// MMA issuer (one warp, one elected lane).  S^T and P^T are double-buffered
// (buffer = tile counter mod 2), so S^T of tile j+1 is issued before P.V of
// tile j and the softmax of tile j+1 overlaps the tensor-core work of tile j:
// per tile, S^T_j = K_j Q^T into buffer j % 2 once the softmax has read S^T_j-2
// out of it, then O^T += V^T_j-1 P^T_j-1 once the softmax has written P^T_j-1.
// The last tile of a work item issues its own P.V before the next item starts,
// so the epilogue never waits for the next item's loads.  A tile of two blocks
// takes two S^T groups (one per block, into the block's columns of the
// buffer) and two P.V groups (one per block, both into O^T).
template <class C, class U>
__device__ void gen_mma(const GenParams &p, const GenSched &sc, uint8_t *smem, GenBars *bars, uint32_t tmem_any) {
    // the whole warp runs this loop converged, with warp-uniform values; one
    // elected lane issues each MMA and commit
    volatile int *abort_flag = &bars->abort;
    const uint32_t tmem = __shfl_sync(0xffffffffu, tmem_any, 0);   // the same in every lane
    constexpr uint32_t kIdS = gen_idesc(C::FMT, false, false);
    constexpr uint32_t kIdPV = gen_idesc(C::FMT, true, true);
    const uint32_t o_tm = tmem + C::O_COL;
    const uint64_t q_desc0 = smem_desc(smem_u32(smem + C::OFF_Q), 16, 1024, 2);
    // P^T: MN-major, one swizzled row of 32 heads per key (64 or 32 bytes)
    const uint64_t p_desc0 = smem_desc(smem_u32(smem + C::OFF_P), C::P_BYTES, 8 * C::P_ROW, C::P_SWZ);
    uint32_t cons = 0, qn = 0;
    bool ok = true;

    // P.V of tile counter j (stage st); `first` starts the item's O^T
    auto issue_pv = [&](uint32_t j, int st, bool first) -> bool {
        const uint32_t b = j & 1;
        if (!warp_wait(smem_u32(&bars->p_full[b]), (j >> 1) & 1, abort_flag)) return false;
        tc_fence_after();
        // O^T: A = V tile MN-major (M = head dim over the panels, LBO = panel
        // stride), B = P^T MN-major (32 heads in one swizzled row per key);
        // each k-step is MMA_K keys
        const uint32_t kaddr = smem_u32(smem + C::OFF_KV + st * C::STAGE_BYTES);
#pragma unroll
        for (int x = 0; x < C::BLK; ++x) {
            const uint64_t v_desc = smem_desc(kaddr + C::TILE_BYTES + x * C::BLK_BYTES, kPanelBytes, 1024, 2);
            const uint64_t p_desc = p_desc0 + (((b * C::BLK + x) * C::P_BYTES) >> 4);
#pragma unroll
            for (int kk = 0; kk < kKT / C::MMA_K; ++kk)
                mma_ss_e<C::FP8>(o_tm, v_desc + ((kk * C::MMA_K * 128) >> 4),
                                 p_desc + ((kk * C::MMA_K * C::P_ROW) >> 4), kIdPV,
                                 (!first || x > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit_e(smem_u32(&bars->pv_done[b]));
        tc_commit_e(smem_u32(&bars->kv_empty[st]));
        return true;
    };

    GenCursor cur;
    while (ok) {
        GenItem it;
        if (!gen_next<U>(p, sc, cur, it, false)) break;
        const int qs = qn % kQSlots;
        if (!warp_wait(smem_u32(&bars->q_full[qs]), (qn / kQSlots) & 1, abort_flag)) break;
        ++qn;
        const uint64_t q_desc = q_desc0 + ((qs * C::Q_BYTES) >> 4);
        bool first = true;
        int prev_st = 0;
        for (int k = it.k0; k < it.k1; k += U::TK) {
            const int st = cons % C::NS;
            const uint32_t b = cons & 1;
            if (!warp_wait(smem_u32(&bars->kv_full[st]), (cons / C::NS) & 1, abort_flag) ||
                (cons >= 2 && !warp_wait(smem_u32(&bars->s_free[b]), ((cons - 2) >> 1) & 1, abort_flag))) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t kaddr = smem_u32(smem + C::OFF_KV + st * C::STAGE_BYTES);
            // S^T: A = K tile (K-major, 128 keys), B = Q tile (K-major, 32 heads);
            // each k-step (16 dims of 16 bits or 32 of 8) is 32 bytes within a
            // 128-byte panel row
#pragma unroll
            for (int x = 0; x < C::BLK; ++x) {
                const uint64_t k_desc = smem_desc(kaddr + x * C::BLK_BYTES, 16, 1024, 2);
#pragma unroll
                for (int kk = 0; kk < kD / C::MMA_K; ++kk) {
                    const uint32_t koff = (kk * 32 / 128) * kPanelBytes + (kk * 32) % 128;
                    const uint32_t qoff = (kk * 32 / 128) * kQPanelBytes + (kk * 32) % 128;
                    mma_ss_e<C::FP8>(tmem + b * C::SCOLS + x * kNP, k_desc + (koff >> 4), q_desc + (qoff >> 4), kIdS,
                                     kk > 0 ? 1u : 0u);
                }
            }
            if (k + U::TK >= it.k1) tc_commit_e(smem_u32(&bars->q_empty[qs]));
            tc_commit_e(smem_u32(&bars->s_full[b]));
            if (!first && !issue_pv(cons - 1, prev_st, k - U::TK == it.k0)) {
                ok = false;
                break;
            }
            prev_st = st;
            first = false;
            ++cons;
        }
        if (!ok) break;
        // the item's last P.V (none for an item without keys), then O^T is complete
        if (!first && !issue_pv(cons - 1, prev_st, it.k1 - it.k0 <= U::TK)) break;
        tc_commit_e(smem_u32(&bars->o_full));
    }
    // no tensor-core operation may be in flight when TMEM is released
    tc_commit_e(smem_u32(&bars->drain));
    mbar_wait_drain(smem_u32(&bars->drain), 0);
}

// Softmax and epilogue.  Softmax warp w owns rows 32 (w % 4) .. + 31 of every
// tile block (its TMEM lanes of S^T) and the same rows of O^T (head
// dimensions).  Row r of block i is key U::row_key(i, r) of kv head
// g + U::row_head(i, r).
//
// Columns of S^T are query heads: [0, G) of a one-head unit, or [0, G) and
// [16, 16 + G) of a two-head unit (its Q tile is two 16-row halves).  A
// thread works on NC >= G columns of each block, from the block's first
// column cb: in a one-block two-head unit (MODE 1) the columns of the row's
// kv head (warps 0-1 the first head, 2-3 the second: one column group per
// head); in a two-block two-head unit columns [0, NC) of block 0 (the first
// head's keys) and [16, 16 + NC) of block 1 (the second's), both in every
// thread; in MODE 2 warps 0-3 and 4-7 take columns 0-15 and 16-31 (two column
// groups); in MODE 0 all four warps take columns [0, NC).  Columns of a group
// past G hold other heads' queries and feed only O^T columns that are never
// stored.  In a two-head unit a row's weights in the other head's columns are
// written as 0, so P.V adds, for each column, only the rows of its own kv
// head.  In a one-block two-head unit an O^T row holds columns of both
// heads' column groups, so the rescale factors and reference maxima of every
// column go through shared memory; elsewhere every thread of a group holds
// the factors of all the columns it rescales.
template <class C, class U, int NC, int MODE>
__device__ void gen_softmax(const GenParams &p, const GenSched &sc, uint8_t *smem, GenBars *bars, uint32_t tmem,
                            int warp, int lane) {
    using L = Layout<MODE>;
    constexpr bool two = U::TWO;
    constexpr int BLK = C::BLK;
    constexpr bool SPLIT_HEADS = two && BLK == 1;       // column groups per head, factors through shared memory
    constexpr int NSET = two && BLK == 2 ? 2 : 1;       // column sets of a thread (one per head of a two-block tile)
    constexpr int ST = L::SW * 32;                      // softmax threads
    constexpr int NW = SPLIT_HEADS ? 2 : 4;             // warps of a column group
    volatile int *abort_flag = &bars->abort;
    const int r = (warp & 3) * 32 + lane;               // block row = TMEM lane
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t o_tm = lane_base + C::O_COL;
    uint8_t *prow0 = smem + C::OFF_P + r * C::P_ROW;     // this row's P^T row in buffer 0, block 0
    const int gi = SPLIT_HEADS ? warp >> 1 : MODE == 2 ? warp >> 2 : 0;   // column group
    const int c0 = 16 * gi;                             // its first column
    const int w0 = gi * NW;                             // its first warp
    // first column of set q (and of block q's values) of this thread
    auto cset = [&](int q) { return NSET == 2 ? 16 * q : c0; };
    // P^T swizzle: 16-byte chunk index ^= (row / 2) % 4 (64-byte rows) or (row / 4) % 2 (32-byte rows)
    const uint32_t swz = C::FP8 ? (r >> 2) & 1 : (r >> 1) & 3;
    uint32_t oph = 0, cons = 0;
    GenCursor cur;
    for (;;) {
        GenItem it;
        if (!gen_next<U>(p, sc, cur, it, false)) break;
        float m[NSET][NC], l[NSET][NC];
#pragma unroll
        for (int q = 0; q < NSET; ++q)
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                m[q][c] = -INFINITY;   // reference max (log2 units) P and O^T are relative to
                l[q][c] = 0.f;         // this thread's part of the row sum
            }
        bool ok = true, first = true;
        for (int k = it.k0; k < it.k1; k += U::TK) {
            // S^T_j and P^T_j use buffer j % 2.  The commit that completes
            // S^T_j also covers P.V_j-2, issued before it by the same thread,
            // so P^T buffer j % 2 is free to rewrite once S^T_j is here.
            const uint32_t b = cons & 1;
            const bool got = mbar_wait(smem_u32(&bars->s_full[b]), (cons >> 1) & 1, abort_flag);
            if (!soft_all<ST>(got)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int st = cons % C::NS;
            const uint32_t j = cons++;
            uint32_t sr[BLK][NC];
#pragma unroll
            for (int i = 0; i < BLK; ++i) tmem_ld_n<NC>(lane_base + b * C::SCOLS + i * kNP + cset(i), sr[i]);
#pragma unroll
            for (int i = 0; i < BLK; ++i) tmem_wait_ld_n<NC>(sr[i]);
            tc_fence_before();
            mbar_arrive(smem_u32(&bars->s_free[b]));   // S^T buffer b may take S^T_j+2
            float s[BLK][NC];
            bool need = false;
#pragma unroll
            for (int i = 0; i < BLK; ++i) {
                const int q = NSET == 2 ? i : 0;
                const bool valid = k + U::row_key(i, r) < it.k1;
#pragma unroll
                for (int c = 0; c < NC; ++c) {
                    s[i][c] = valid ? __uint_as_float(sr[i][c]) * p.c : -INFINITY;
                    need |= s[i][c] > m[q][c] + kRescaleLog2;
                }
            }
            bool rescaled = false;
            if (soft_any<ST>(need)) {
                // tile maximum of every column over the group's rows
#pragma unroll
                for (int q = 0; q < NSET; ++q)
#pragma unroll
                    for (int c = 0; c < NC; ++c) {
                        float x = s[q][c];
                        if constexpr (NSET == 1 && BLK == 2) x = fmaxf(x, s[1][c]);
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
                        if (lane == 0) bars->red[warp][cset(q) + c] = x;
                    }
                soft_sync<ST>();
                float alpha[NSET][NC];
#pragma unroll
                for (int q = 0; q < NSET; ++q)
#pragma unroll
                    for (int c = 0; c < NC; ++c) {
                        const int col = cset(q) + c;
                        float tmax = fmaxf(bars->red[w0][col], bars->red[w0 + 1][col]);
                        if (NW == 4) tmax = fmaxf(tmax, fmaxf(bars->red[w0 + 2][col], bars->red[w0 + 3][col]));
                        alpha[q][c] = 1.f;
                        if (tmax > m[q][c] + kRescaleLog2) {
                            alpha[q][c] = m[q][c] == -INFINITY ? 0.f : ex2(m[q][c] - tmax);
                            l[q][c] *= alpha[q][c];
                            m[q][c] = tmax;
                        }
                    }
                if (SPLIT_HEADS && !first && warp == w0 && lane == 0) {
#pragma unroll
                    for (int c = 0; c < NC; ++c) bars->alpha[c0 + c] = alpha[0][c];
                }
                soft_sync<ST>();   // the scratch rows may be rewritten after this
                if (!first) {
                    // O^T holds the P.V of the previous tile once it is done
                    const bool pv = mbar_wait(smem_u32(&bars->pv_done[(j - 1) & 1]), ((j - 1) >> 1) & 1, abort_flag);
                    if (!soft_all<ST>(pv)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if constexpr (SPLIT_HEADS) {
                        // row r of O^T holds both heads' columns
                        uint32_t orr[32];
                        tmem_ld32(o_tm, orr);
                        tmem_wait_ld(orr);
#pragma unroll
                        for (int h = 0; h < kNP; ++h)
                            orr[h] = __float_as_uint(__uint_as_float(orr[h]) * bars->alpha[h]);
                        tmem_st32(o_tm, orr);
                        soft_sync<ST>();   // every thread has read the factors
                    } else {
                        // this thread's columns of row r of O^T
#pragma unroll
                        for (int q = 0; q < NSET; ++q) {
                            uint32_t orr[NC];
                            tmem_ld_n<NC>(o_tm + cset(q), orr);
                            tmem_wait_ld_n<NC>(orr);
#pragma unroll
                            for (int c = 0; c < NC; ++c)
                                orr[c] = __float_as_uint(__uint_as_float(orr[c]) * alpha[q][c]);
                            tmem_st_n<NC>(o_tm + cset(q), orr);
                        }
                    }
                    rescaled = true;
                }
            }
            float pv[BLK][NC];
#pragma unroll
            for (int i = 0; i < BLK; ++i) {
                const int q = NSET == 2 ? i : 0;
#pragma unroll
                for (int c = 0; c < NC; ++c) {
                    pv[i][c] = m[q][c] == -INFINITY ? 0.f : ex2(s[i][c] - m[q][c]);
                    l[q][c] += pv[i][c];
                }
            }
#pragma unroll
            for (int i = 0; i < BLK; ++i) {
                // P^T row r of block i: columns [cb, cb + NC) from pv and, in
                // a two-head unit, 0 in the other head's columns (the
                // remaining columns feed only O^T columns that are never
                // stored)
                uint8_t *prow = prow0 + (b * BLK + i) * C::P_BYTES;
                constexpr int VB = NC * C::E;                    // bytes of this thread's values
                uint32_t w[(VB + 3) / 4];
                if constexpr (C::FP8) {
#pragma unroll
                    for (int x = 0; x < NC / 4; ++x)
                        w[x] = pack4_e4m3(pv[i][4 * x], pv[i][4 * x + 1], pv[i][4 * x + 2], pv[i][4 * x + 3]);
                } else {
#pragma unroll
                    for (int x = 0; x < NC / 2; ++x) w[x] = pack2<C::FMT == 1u>(pv[i][2 * x], pv[i][2 * x + 1]);
                }
                const int cb = cset(NSET == 2 ? i : 0);
                const int vo = cb * C::E;                    // byte offset of the values in the row
                const int zo = (16 - cb) * C::E;             // the other head's columns
                if constexpr (VB >= 16) {
#pragma unroll
                    for (int c = 0; c < VB / 16; ++c) {
                        *reinterpret_cast<uint4 *>(prow + ((((vo >> 4) + c) ^ swz) << 4)) =
                            make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
                        if (two)
                            *reinterpret_cast<uint4 *>(prow + ((((zo >> 4) + c) ^ swz) << 4)) = make_uint4(0u, 0u, 0u, 0u);
                    }
                } else if constexpr (VB == 8) {
                    *reinterpret_cast<uint2 *>(prow + ((((vo >> 4) ^ swz) << 4) | (vo & 15))) = make_uint2(w[0], w[1]);
                    if (two) *reinterpret_cast<uint2 *>(prow + ((((zo >> 4) ^ swz) << 4) | (zo & 15))) = make_uint2(0u, 0u);
                } else {
                    static_assert(VB == 4, "P^T values of a thread");
                    *reinterpret_cast<uint32_t *>(prow + ((((vo >> 4) ^ swz) << 4) | (vo & 15))) = w[0];
                    if (two) *reinterpret_cast<uint32_t *>(prow + ((((zo >> 4) ^ swz) << 4) | (zo & 15))) = 0u;
                }
                if (k + U::row_key(i, r) >= it.k1 && (MODE != 2 || gi == 0)) {
                    // a row whose key is past the chunk's end: its V row (stale
                    // cache contents, possibly not finite) is zeroed so that P = 0
                    // contributes 0 (by one column group of the row)
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    uint8_t *vrow = smem + C::OFF_KV + st * C::STAGE_BYTES + C::TILE_BYTES + i * C::BLK_BYTES + r * 128;
#pragma unroll
                    for (int pn = 0; pn < C::PANELS; ++pn)
#pragma unroll
                        for (int c = 0; c < 8; ++c)
                            *reinterpret_cast<uint4 *>(vrow + pn * kPanelBytes + ((c ^ (r & 7)) << 4)) =
                                make_uint4(0u, 0u, 0u, 0u);
                }
            }
            // generic-proxy writes (P^T, zeroed V rows) become visible to the
            // tensor core; TMEM stores complete; then publish
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            if (rescaled) tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bars->p_full[b]));
            first = false;
        }
        if (!ok) break;

        // epilogue: row sums of every column, then the normalised partial O
        // and its LSE
        const bool got = mbar_wait(smem_u32(&bars->o_full), oph, abort_flag);
        oph ^= 1;
        if (!soft_all<ST>(got)) break;
        tc_fence_after();
#pragma unroll
        for (int q = 0; q < NSET; ++q)
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                float x = l[q][c];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
                if (lane == 0) bars->red[warp][cset(q) + c] = x;
            }
        if (SPLIT_HEADS && warp == w0 && lane == 0) {
#pragma unroll
            for (int c = 0; c < NC; ++c) bars->mref[c0 + c] = m[0][c];
        }
        soft_sync<ST>();
        const int64_t row0 = (int64_t)it.b * p.H + (int64_t)it.g * p.G;
        if constexpr (SPLIT_HEADS) {
            // row r of O^T: column h is query head row0 + G * (h / 16) + h % 16
            uint32_t orr[32];
            tmem_ld32(o_tm, orr);
            tmem_wait_ld(orr);
#pragma unroll
            for (int h = 0; h < kNP; ++h) {
                if ((h & 15) < NC && (h & 15) < p.G) {
                    const int g2 = 2 * (h >> 4);
                    const float lt = bars->red[g2][h] + bars->red[g2 + 1][h];
                    const int64_t slot = (row0 + (h >> 4) * p.G + (h & 15)) * p.max_seg + it.seg;
                    p.part_o[slot * kD + r] = lt > 0.f ? __uint_as_float(orr[h]) / lt : 0.f;
                    if (r == h) p.part_lse[slot] = lt > 0.f ? (bars->mref[h] + log2f(lt)) * kLn2 : -INFINITY;
                }
            }
        } else {
            // this thread's columns of row r of O^T
            if constexpr (NSET == 1) {
                // column c0 + c is query head row0 + c0 + c
                uint32_t orr[NC];
                tmem_ld_n<NC>(o_tm + c0, orr);
                tmem_wait_ld_n<NC>(orr);
#pragma unroll
                for (int c = 0; c < NC; ++c) {
                    if (c0 + c < p.G) {
                        const float lt = (bars->red[w0][c0 + c] + bars->red[w0 + 1][c0 + c]) +
                                         (bars->red[w0 + 2][c0 + c] + bars->red[w0 + 3][c0 + c]);
                        const int64_t slot = (row0 + c0 + c) * p.max_seg + it.seg;
                        p.part_o[slot * kD + r] = lt > 0.f ? __uint_as_float(orr[c]) / lt : 0.f;
                        if (r == c) p.part_lse[slot] = lt > 0.f ? (m[0][c] + log2f(lt)) * kLn2 : -INFINITY;
                    }
                }
            } else {
                // column 16 q + c is query head row0 + q * G + c (all four warps)
#pragma unroll
                for (int q = 0; q < NSET; ++q) {
                    uint32_t orr[NC];
                    tmem_ld_n<NC>(o_tm + 16 * q, orr);
                    tmem_wait_ld_n<NC>(orr);
#pragma unroll
                    for (int c = 0; c < NC; ++c) {
                        const int col = 16 * q + c;
                        if (c < p.G) {
                            const float lt = (bars->red[0][col] + bars->red[1][col]) + (bars->red[2][col] + bars->red[3][col]);
                            const int64_t slot = (row0 + q * p.G + c) * p.max_seg + it.seg;
                            p.part_o[slot * kD + r] = lt > 0.f ? __uint_as_float(orr[c]) / lt : 0.f;
                            if (r == col) p.part_lse[slot] = lt > 0.f ? (m[q][c] + log2f(lt)) * kLn2 : -INFINITY;
                        }
                    }
                }
            }
        }
        soft_sync<ST>();   // the scratch rows may be rewritten after this
    }
}

template <int ELEM, int NC, int MODE>
__global__ void __launch_bounds__(Layout<MODE>::THREADS, 1)
    fmha_gen_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const GenParams p) {
    using L = Layout<MODE>;
    using C = GenCfg<ELEM, GenBlk<ELEM, MODE>::value>;
    using U = Unit<L::TWO, C::BLK>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    GenBars *bars = reinterpret_cast<GenBars *>(smem + C::OFF_BARS);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kQSlots; ++i) {
            mbar_init(smem_u32(&bars->q_full[i]), 1);
            mbar_init(smem_u32(&bars->q_empty[i]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&bars->s_full[b]), 1);
            mbar_init(smem_u32(&bars->s_free[b]), L::SW * 32);
            mbar_init(smem_u32(&bars->p_full[b]), L::SW);
            mbar_init(smem_u32(&bars->pv_done[b]), 1);
        }
        mbar_init(smem_u32(&bars->o_full), 1);
        mbar_init(smem_u32(&bars->drain), 1);
        for (int s = 0; s < kNSMax; ++s) {
            mbar_init(smem_u32(&bars->kv_full[s]), 1);
            mbar_init(smem_u32(&bars->kv_empty[s]), 1);
        }
        bars->abort = 0;
        for (int i = 0; i < kNP; ++i) bars->alpha[i] = 1.f;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == L::MMA) {
        tmem_alloc(smem_u32(&bars->tmem_base), C::TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == L::PROD) gen_schedule<U>(p, &bars->sched, lane);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    // the merge kernel may be scheduled as CTAs of this grid exit; it waits
    // for this grid's completion before it reads the partials
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const GenSched sc = bars->sched;
    if (warp < L::SW) {
        gen_softmax<C, U, NC, MODE>(p, sc, smem, bars, tmem, warp, lane);
    } else if (warp == L::PROD) {
        if (lane == 0) gen_producer<C, U>(p, sc, &tmQ, &tmK, &tmV, smem, bars);
    } else {
        gen_mma<C, U>(p, sc, smem, bars, tmem);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == L::MMA) {
        __syncwarp();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// One CTA of kMergeThreads per (sequence, query head), for rows merged from
// many chunks (eight warps share them): O = out_scale *
// sum_c w_c O_c / sum_c w_c with w_c = exp(LSE_c - max LSE), LSE = max +
// ln sum_c w_c.  Eight groups of 32 threads take every eighth chunk (each
// thread four of the 128 dims), so eight 512-byte partial rows are in flight.
constexpr int kMergeThreads = 256;
constexpr int kMergeGroups = kMergeThreads / 32;

template <int ELEM>
__global__ void __launch_bounds__(kMergeThreads) fmha_gen_merge_block_kernel(const GenParams p) {
    __shared__ float red_m[kMergeGroups];
    __shared__ float4 red_o[kMergeGroups][32];
    __shared__ float red_w[kMergeGroups];
    __shared__ long long red_t[kMergeGroups], red_p[kMergeGroups];
    const int row = blockIdx.x;
    const int grp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = row / p.H, u = (row % p.H) / (p.G * p.GP);   // sequence and work unit
    // the attention kernel's split: total tiles, and the tiles before sequence b
    long long tot = 0, pre = 0;
    for (int bb = threadIdx.x; bb < p.B; bb += kMergeThreads) {
        const long long n = (long long)p.NU * gen_tiles(p, bb, p.TK);
        tot += n;
        if (bb < b) pre += n;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        tot += __shfl_xor_sync(0xffffffffu, tot, o);
        pre += __shfl_xor_sync(0xffffffffu, pre, o);
    }
    if (lane == 0) {
        red_t[grp] = tot;
        red_p[grp] = pre;
    }
    __syncthreads();
    tot = 0;
    pre = 0;
#pragma unroll
    for (int i = 0; i < kMergeGroups; ++i) {
        tot += red_t[i];
        pre += red_p[i];
    }
    const int nt = gen_tiles(p, b, p.TK);
    int nch = 0;                       // CTAs that covered this pair = its partial slots
    if (nt > 0) {
        const long long per = (tot + p.ncta - 1) / p.ncta;
        const long long off = pre + (long long)u * nt;
        nch = (int)((off + nt - 1) / per - off / per + 1);
    }
    // the partials are the attention kernel's: wait for it (and its memory)
    // here; everything above overlaps its tail
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const float *lse_c = p.part_lse + (int64_t)row * p.max_seg;
    float mx = -INFINITY;
    for (int c = threadIdx.x; c < nch; c += kMergeThreads) mx = fmaxf(mx, lse_c[c]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) red_m[grp] = mx;
    __syncthreads();
    mx = red_m[0];
#pragma unroll
    for (int i = 1; i < kMergeGroups; ++i) mx = fmaxf(mx, red_m[i]);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float wsum = 0.f;
    if (mx != -INFINITY) {
        for (int c = grp; c < nch; c += kMergeGroups) {
            const float w = __expf(lse_c[c] - mx);
            const float4 v =
                *reinterpret_cast<const float4 *>(p.part_o + ((int64_t)row * p.max_seg + c) * kD + lane * 4);
            wsum += w;
            acc.x += w * v.x;
            acc.y += w * v.y;
            acc.z += w * v.z;
            acc.w += w * v.w;
        }
    }
    red_o[grp][lane] = acc;
    if (lane == 0) red_w[grp] = wsum;
    __syncthreads();
    if (grp != 0) return;
    for (int i = 1; i < kMergeGroups; ++i) {
        const float4 v = red_o[i][lane];
        acc.x += v.x;
        acc.y += v.y;
        acc.z += v.z;
        acc.w += v.w;
        wsum += red_w[i];
    }
    if (lane != 0) wsum = 0.f;   // lane 0 holds group 0's sum; share the total
    wsum = __shfl_sync(0xffffffffu, lane == 0 ? wsum : 0.f, 0);
    const float inv = wsum > 0.f ? p.out_scale / wsum : 0.f;
    if constexpr (ELEM == FMHA_E4M3) {
        *reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(p.o) + (int64_t)row * kD + lane * 4) =
            pack4_e4m3(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    } else {
        uint2 out;
        out.x = pack2<ELEM == FMHA_BF16>(acc.x * inv, acc.y * inv);
        out.y = pack2<ELEM == FMHA_BF16>(acc.z * inv, acc.w * inv);
        *reinterpret_cast<uint2 *>(static_cast<uint16_t *>(p.o) + (int64_t)row * kD + lane * 4) = out;
    }
    if (lane == 0 && p.lse) p.lse[row] = wsum > 0.f ? mx + __logf(wsum) : -INFINITY;
}

// One warp per (sequence, query head) row, blockDim / 32 rows per CTA (the host
// keeps at least two CTAs per SM): O = out_scale *
// sum_c w_c O_c / sum_c w_c with w_c = exp(LSE_c - max LSE), LSE = max +
// ln sum_c w_c.  Lane l holds dims 4l .. 4l + 3; no shared memory and no
// block barrier, so after the wait a row of at most eight chunks is one round
// of loads (its chunks' LSEs and partial rows together) and a store.
constexpr int kMergeRowsMax = 8;

template <int ELEM>
__global__ void __launch_bounds__(32 * kMergeRowsMax) fmha_gen_merge_warp_kernel(const GenParams p) {
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (row >= p.B * p.H) return;
    const int b = row / p.H, u = (row % p.H) / (p.G * p.GP);   // sequence and work unit
    // the attention kernel's split: total tiles, and the tiles before sequence b
    long long tot = 0, pre = 0;
    for (int bb = lane; bb < p.B; bb += 32) {
        const long long n = (long long)p.NU * gen_tiles(p, bb, p.TK);
        tot += n;
        if (bb < b) pre += n;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        tot += __shfl_xor_sync(0xffffffffu, tot, o);
        pre += __shfl_xor_sync(0xffffffffu, pre, o);
    }
    const int nt = gen_tiles(p, b, p.TK);
    int nch = 0;                       // CTAs that covered this unit = its partial slots
    if (nt > 0) {
        const long long per = (tot + p.ncta - 1) / p.ncta;
        const long long off = pre + (long long)u * nt;
        nch = (int)((off + nt - 1) / per - off / per + 1);
    }
    // the partials are the attention kernel's: wait for it (and its memory)
    // here; everything above overlaps its tail
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const float *lse_c = p.part_lse + (int64_t)row * p.max_seg;
    const float4 *o_c = reinterpret_cast<const float4 *>(p.part_o + (int64_t)row * p.max_seg * kD) + lane;
    // the first 32 chunks' LSEs and the first eight chunks' partial rows go
    // out together: one memory round trip for a row of at most eight chunks
    const float lse0 = lane < nch ? lse_c[lane] : -INFINITY;
    float4 v0[8];
#pragma unroll
    for (int x = 0; x < 8; ++x) v0[x] = x < nch ? o_c[(int64_t)x * (kD / 4)] : make_float4(0.f, 0.f, 0.f, 0.f);
    float mx = lse0;
    for (int c = 32 + lane; c < nch; c += 32) mx = fmaxf(mx, lse_c[c]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float wsum = 0.f;
    if (mx != -INFINITY) {
        for (int c0 = 0; c0 < nch; c0 += 32) {
            // weights of 32 chunks at a time, one per lane, then broadcast
            const float wl = c0 + lane < nch ? __expf((c0 == 0 ? lse0 : lse_c[c0 + lane]) - mx) : 0.f;
            const int cn = nch - c0 < 32 ? nch - c0 : 32;
            // eight chunks' rows in flight at a time
            for (int c = 0; c < cn; c += 8) {
                float4 v[8];
#pragma unroll
                for (int x = 0; x < 8; ++x)
                    v[x] = c0 + c == 0 ? v0[x]
                                       : c + x < cn ? o_c[(int64_t)(c0 + c + x) * (kD / 4)] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int x = 0; x < 8; ++x) {
                    const float w = __shfl_sync(0xffffffffu, wl, (c + x) & 31);
                    if (c + x < cn) {
                        wsum += w;
                        acc.x += w * v[x].x;
                        acc.y += w * v[x].y;
                        acc.z += w * v[x].z;
                        acc.w += w * v[x].w;
                    }
                }
            }
        }
    }
    const float inv = wsum > 0.f ? p.out_scale / wsum : 0.f;
    if constexpr (ELEM == FMHA_E4M3) {
        *reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(p.o) + (int64_t)row * kD + lane * 4) =
            pack4_e4m3(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    } else {
        uint2 out;
        out.x = pack2<ELEM == FMHA_BF16>(acc.x * inv, acc.y * inv);
        out.y = pack2<ELEM == FMHA_BF16>(acc.z * inv, acc.w * inv);
        *reinterpret_cast<uint2 *>(static_cast<uint16_t *>(p.o) + (int64_t)row * kD + lane * 4) = out;
    }
    if (lane == 0 && p.lse) p.lse[row] = wsum > 0.f ? mx + __logf(wsum) : -INFINITY;
}

PFN_cuTensorMapEncodeTiled_v12000 gen_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
        else
            cudaGetLastError();
    });
    return fn;
}

int gen_sm_count() {
    static std::mutex mu;
    static int cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
    std::lock_guard<std::mutex> lk(mu);
    if (cached[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
        cached[dev] = n;
    }
    return cached[dev];
}

}  // namespace

int gen_set_wait_limit(unsigned long long ns) {
    const unsigned long long v = ns ? ns : kTimeoutNs;
    if (cudaMemcpyToSymbol(g_gen_wait_ns, &v, sizeof(v)) != cudaSuccess) {
        cudaGetLastError();
        return FMHA_ERR_CUDA;
    }
    return FMHA_OK;
}

int gen_set_test_gate(int on) {
    const int v = on ? 1 : 0;
    if (cudaMemcpyToSymbol(g_gen_test_gate, &v, sizeof(v)) != cudaSuccess) {
        cudaGetLastError();
        return FMHA_ERR_CUDA;
    }
    return FMHA_OK;
}

int gen_read_status(int reset) {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_gen_status, sizeof(int)) != cudaSuccess) return FMHA_ERR_CUDA;
    if (reset && v != 0) {
        const int z = 0;
        if (cudaMemcpyToSymbol(g_gen_status, &z, sizeof(int)) != cudaSuccess) return FMHA_ERR_CUDA;
    }
    return v;
}

}  // namespace fmha

using namespace fmha;

namespace {

struct GenLayout {
    int max_seg;
    size_t o_bytes, lse_off, total;
};

// Instantiations: two-head units with 4, 8 or 16 columns per thread (G <= 16);
// one-head units with 8 or 16 (G <= 16), or two groups of 16 (G > 16).
using GenKernel = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, GenParams);
template <int ELEM>
GenKernel gen_kernel_nc(int nc, int mode) {
    if (mode == 1)
        return nc == 4 ? fmha_gen_kernel<ELEM, 4, 1>
               : nc == 8 ? fmha_gen_kernel<ELEM, 8, 1> : fmha_gen_kernel<ELEM, 16, 1>;
    if (mode == 2) return fmha_gen_kernel<ELEM, 16, 2>;
    return nc == 8 ? fmha_gen_kernel<ELEM, 8, 0> : fmha_gen_kernel<ELEM, 16, 0>;
}
GenKernel gen_kernel_for(int dt, int nc, int mode) {
    return dt == FMHA_BF16 ? gen_kernel_nc<FMHA_BF16>(nc, mode)
           : dt == FMHA_F16 ? gen_kernel_nc<FMHA_F16>(nc, mode) : gen_kernel_nc<FMHA_E4M3>(nc, mode);
}

// Two adjacent kv heads share a work unit when H_k is even and each query
// group fits a 16-column half of S^T.
bool gen_pairs(int H, int H_k) { return H_k % 2 == 0 && 2 * (H / H_k) <= kNP; }

// Tile blocks and shared memory of the kernel for an element type and warp layout
template <int ELEM>
int gen_blocks_t(int mode) {
    return mode == 1 ? GenBlk<ELEM, 1>::value : mode == 2 ? GenBlk<ELEM, 2>::value : GenBlk<ELEM, 0>::value;
}
int gen_blocks(int dt, int mode) {
    return dt == FMHA_BF16 ? gen_blocks_t<FMHA_BF16>(mode)
           : dt == FMHA_F16 ? gen_blocks_t<FMHA_F16>(mode) : gen_blocks_t<FMHA_E4M3>(mode);
}
template <int ELEM>
int gen_smem_t(int mode) {
    return mode == 1   ? GenCfg<ELEM, GenBlk<ELEM, 1>::value>::SMEM_BYTES
           : mode == 2 ? GenCfg<ELEM, GenBlk<ELEM, 2>::value>::SMEM_BYTES
                       : GenCfg<ELEM, GenBlk<ELEM, 0>::value>::SMEM_BYTES;
}
int gen_smem_bytes(int dt, int mode) {
    return dt == FMHA_BF16 ? gen_smem_t<FMHA_BF16>(mode)
           : dt == FMHA_F16 ? gen_smem_t<FMHA_F16>(mode) : gen_smem_t<FMHA_E4M3>(mode);
}

// Partial slots per (sequence, head): a unit of n tiles meets at most n + 1
// CTAs' ranges, and n <= ceil(S_max / keys per tile).
GenLayout gen_layout(int B, int H, int H_k, int S_max) {
    GenLayout g;
    const int tk = gen_pairs(H, H_k) ? kKT / 2 : kKT;
    g.max_seg = (S_max + tk - 1) / tk + 1;
    const size_t rows = (size_t)B * H * g.max_seg;
    g.o_bytes = rows * kD * sizeof(float);
    g.lse_off = (g.o_bytes + 255) / 256 * 256;
    g.total = g.lse_off + rows * sizeof(float);
    return g;
}

}  // namespace

extern "C" size_t fmha_gen_workspace_size(int B, int H, int H_k, int D, int S_max) {
    if (B <= 0 || H <= 0 || H_k <= 0 || H % H_k != 0 || D != kD || S_max <= 0) return 0;
    return gen_layout(B, H, H_k, S_max).total;
}

extern "C" int fmha_gen_fwd(fmha_tensor q, fmha_tensor k_cache, fmha_tensor v_cache, fmha_tensor k_new,
                            fmha_tensor v_new, fmha_tensor o, float *lse, int B, int H, int H_k, int D, int B_cache,
                            int S_max, const int *seqlen, const int *batch_idx, float scale, float out_scale,
                            void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    // ---- host-side validation: nothing is launched on a bad argument ----
    if (B < 0 || H <= 0 || H_k <= 0 || H % H_k != 0 || H / H_k > kNP || D != kD) return FMHA_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !(scale < INFINITY) || !(out_scale == out_scale) || out_scale == INFINITY ||
        out_scale == -INFINITY)
        return FMHA_ERR_INVALID_ARG;
    if ((k_new.data == nullptr) != (v_new.data == nullptr)) return FMHA_ERR_INVALID_ARG;
    const bool insert = k_new.data != nullptr;
    if (B == 0) return FMHA_OK;
    if (S_max <= 0 || B_cache <= 0 || !seqlen) return FMHA_ERR_INVALID_ARG;
    if (!q.data || !k_cache.data || !v_cache.data || !o.data) return FMHA_ERR_INVALID_ARG;
    const int dt = q.dtype;
    if (dt != FMHA_F16 && dt != FMHA_BF16 && dt != FMHA_E4M3) return FMHA_ERR_UNSUPPORTED;
    if (k_cache.dtype != dt || v_cache.dtype != dt || o.dtype != dt) return FMHA_ERR_UNSUPPORTED;
    if (insert && (k_new.dtype != dt || v_new.dtype != dt)) return FMHA_ERR_UNSUPPORTED;
    auto misaligned = [](const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) != 0; };
    if (misaligned(q.data) || misaligned(k_cache.data) || misaligned(v_cache.data) || misaligned(o.data) ||
        (insert && (misaligned(k_new.data) || misaligned(v_new.data))))
        return FMHA_ERR_UNSUPPORTED;
    if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return FMHA_ERR_INVALID_ARG;
    const GenLayout g = gen_layout(B, H, H_k, S_max);
    const int sms = gen_sm_count();
    if (sms <= 0) return FMHA_ERR_CUDA;
    if (!workspace || workspace_bytes < g.total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return FMHA_ERR_INVALID_ARG;

    GenParams p{};
    p.q = q.data;
    p.k_new = k_new.data;
    p.v_new = v_new.data;
    p.k_cache = k_cache.data;
    p.v_cache = v_cache.data;
    p.seqlen = seqlen;
    p.batch_idx = batch_idx;
    p.o = o.data;
    p.lse = lse;
    p.part_o = static_cast<float *>(workspace);
    p.part_lse = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + g.lse_off);
    p.B = B;
    p.H = H;
    p.H_k = H_k;
    p.G = H / H_k;
    p.GP = gen_pairs(H, H_k) ? 2 : 1;
    // warp layout, and the columns of S^T a softmax thread works on (the
    // query group rounded up; 16 per column group for groups wider than 16)
    const int G = H / H_k;
    const int mode = p.GP == 2 ? 1 : G > 16 ? 2 : 0;
    const int nc = mode == 1 && G <= 4 ? 4 : G <= 8 ? 8 : 16;
    const int blk = gen_blocks(dt, mode);
    p.TK = kKT * blk / p.GP;
    p.NU = H_k / p.GP;
    p.B_cache = B_cache;
    p.S_max = S_max;
    p.max_seg = g.max_seg;
    p.ncta = sms;
    p.insert = insert ? 1 : 0;
    p.dtype = dt;
    p.c = scale * kLog2e;
    p.out_scale = out_scale;

    // ---- tensor maps ----
    auto fn = gen_encode_fn();
    if (!fn) return FMHA_ERR_CUDA;
    const CUtensorMapDataType tdt = dt == FMHA_BF16  ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                    : dt == FMHA_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                     : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    const int esz = dt == FMHA_E4M3 ? 1 : 2;
    const cuuint32_t box_d = 128 / esz;                 // elements of one 128-byte swizzle panel
    CUtensorMap tq, tk, tv;
    {
        // q as [B*H rows, 128]: a box of 32 heads (16 for a two-head unit's
        // halves) x one swizzle panel of dims
        cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)B * H};
        cuuint64_t strides[1] = {(cuuint64_t)kD * esz};
        cuuint32_t box[2] = {box_d, (cuuint32_t)(kNP / p.GP)};
        cuuint32_t es[2] = {1, 1};
        if (fn(&tq, tdt, 2, const_cast<void *>(q.data), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return FMHA_ERR_CUDA;
    }
    for (int kv = 0; kv < 2; ++kv) {
        // cache as [B_cache, S_max, H_k, 128]: a box of the tokens of one
        // head in one tile block (128; 64 in a one-block two-head tile) x
        // one panel
        cuuint64_t dims[4] = {(cuuint64_t)kD, (cuuint64_t)H_k, (cuuint64_t)S_max, (cuuint64_t)B_cache};
        cuuint64_t strides[3] = {(cuuint64_t)kD * esz, (cuuint64_t)kD * esz * H_k,
                                 (cuuint64_t)kD * esz * H_k * S_max};
        cuuint32_t box[4] = {box_d, 1, (cuuint32_t)(blk == 2 ? kKT : p.TK), 1};
        cuuint32_t es[4] = {1, 1, 1, 1};
        if (fn(kv ? &tv : &tk, tdt, 4, kv ? v_cache.data : k_cache.data, dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return FMHA_ERR_CUDA;
    }

    // ---- launch: persistent CTAs over the work items, then the merge ----
    const int grid = sms;   // one persistent CTA per SM; each streams 1/grid of the tiles
    const int threads = mode == 2 ? Layout<2>::THREADS : Layout<0>::THREADS;
    auto kern = gen_kernel_for(dt, nc, mode);
    const int smem_bytes = gen_smem_bytes(dt, mode);
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes) != cudaSuccess)
        return FMHA_ERR_CUDA;
    kern<<<grid, threads, smem_bytes, stream>>>(tq, tk, tv, p);
    if (cudaGetLastError() != cudaSuccess) return FMHA_ERR_CUDA;
    const int rows = B * H;
    // a row meets about sms / (B * units per sequence) + 1 chunks: many chunks
    // go to eight warps per row, few to one warp per row
    const bool many = sms >= 4 * B * p.NU;
    auto merge = many ? (dt == FMHA_BF16 ? fmha_gen_merge_block_kernel<FMHA_BF16>
                         : dt == FMHA_F16 ? fmha_gen_merge_block_kernel<FMHA_F16> : fmha_gen_merge_block_kernel<FMHA_E4M3>)
                      : (dt == FMHA_BF16 ? fmha_gen_merge_warp_kernel<FMHA_BF16>
                         : dt == FMHA_F16 ? fmha_gen_merge_warp_kernel<FMHA_F16> : fmha_gen_merge_warp_kernel<FMHA_E4M3>);
    // launched as a programmatic dependent of the attention kernel, so its
    // launch and prologue overlap that kernel's tail
    cudaLaunchConfig_t cfg = {};
    // rows per CTA (one warp each): as many as keep two CTAs per SM busy, at most eight
    const int rpc = rows / (2 * sms) < 1 ? 1 : rows / (2 * sms) > kMergeRowsMax ? kMergeRowsMax : rows / (2 * sms);
    cfg.gridDim = many ? dim3(rows) : dim3((rows + rpc - 1) / rpc);
    cfg.blockDim = many ? dim3(kMergeThreads) : dim3(32 * rpc);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, merge, p) != cudaSuccess) return FMHA_ERR_CUDA;
    return FMHA_OK;
}
