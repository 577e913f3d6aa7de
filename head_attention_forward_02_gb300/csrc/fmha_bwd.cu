// fmha_bwd.cu -- backward pass of the fused attention forward on sm_103a:
// dQ, dK and dV from dO, the forward's O and its log-sum-exp.
//
// Definition ("CUTLASS Blackwell FMHA 示例完全解析", §FMHA for Blackwell 反向
// (Backward)): with P = softmax(scale Q K^T + mask) and O = P V, per (b, h)
//     D_i   = dO_i . O_i                       (the row sums of O * dO)
//     P_ij  = exp(scale q_i . k_j - LSE_i)     (LSE from the forward pass)
//     dP_ij = dO_i . v_j ,   dS_ij = P_ij (dP_ij - D_i)
//     dQ_i  = scale sum_j dS_ij k_j ,  dK_j = scale sum_i dS_ij q_i ,
//     dV_j  = sum_i P_ij dO_i .
// The page describes three kernels (row sums of O * dO; the main kernel,
// itself split into a dK/dV kernel and a dQ kernel; a dQ conversion), Q and
// K blocking of 128, TMA loads, causal masking (a key past the query's
// position plus the q-offset, or outside the problem, is masked), head dims
// 64 and 128, and no GQA.
//
// This file: a row-sum kernel, then two tcgen05 kernels that each recompute
// S and dP for their tiles, so that every output tile has one owner and no
// atomics are needed.  The dQ kernel owns a 128-row Q tile and loops over key
// tiles: S = Q K^T and dP = dO V^T (both A and B K-major from shared memory)
// land in TMEM; eight warps (one query row per thread, two warps per row
// quadrant) form dS into a separate TMEM buffer as 16-bit values; dQ += dS K
// is a TMEM-A MMA with K read MN-major.  The dK/dV kernel owns a 128-key tile
// and loops over query tiles in halves of 64: S^T = K Q^T and dP^T = V dO^T;
// one key per thread; P^T and dS^T go back over S^T and dP^T; dV += P^T dO and
// dK += dS^T Q.  Each kernel writes its output in the input type directly (no
// fp32 dQ round trip).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <mutex>

#include "fmha_common.h"

namespace fmha {

__device__ int g_bwd_status;   // FMHA_OK, or FMHA_ERR_TIMEOUT after a bounded wait expired
// the bounded waits' limit (ns); set from the host through fmha_set_wait_limit_ns
__device__ unsigned long long g_bwd_wait_ns = 4000000000ull;
// test hook (fmha_set_test_gate): when set, the producer warp first waits for
// a flag that nothing writes, so that bounded wait runs out before any copy
__device__ int g_bwd_test_gate;
__device__ int g_bwd_test_flag;   // never written

namespace {

constexpr int kT = 128;                 // rows per tile, both sides
constexpr int kCompWarps = 8;           // warps 0-7: elementwise work and epilogue
constexpr int kProdWarp = 8;            // TMA producer (the warp waits together, lane 0 issues the copies)
constexpr int kMmaWarp = 9;             // tcgen05.mma issuer (whole warp, one elected lane), owns TMEM
constexpr int kMmaWarp2 = 10;           // dK/dV kernel: issuer of query half b
constexpr int kThreads = 352;
static_assert(kThreads == 32 * (kMmaWarp2 + 1), "one warp per role");
constexpr uint32_t kTmemCols = 512;
constexpr unsigned long long kTimeoutNs = 4000000000ull;   // the default wait limit
constexpr unsigned long long kDrainNs = 200000000ull;
constexpr float kLog2e = 1.4426950408889634f;

enum Mode { kDQ = 0, kDKDV = 1 };

template <int D_, int MODE_>
struct BCfg {
    static constexpr int D = D_;
    static constexpr int ROW = D * 2;                       // bytes per row (16-bit types)
    static constexpr int SW = ROW >= 128 ? 128 : ROW;       // swizzle span
    static constexpr int PANELS = ROW / SW;
    static constexpr int BOX_D = SW / 2;
    static constexpr int PANEL_BYTES = kT * SW;
    static constexpr int TILE_BYTES = kT * ROW;
    static constexpr uint64_t SW_CODE = SW == 128 ? 2 : 4;  // 128-byte or 64-byte swizzle
    static constexpr int SBO = 8 * SW;
    static constexpr int OWN = 0;                           // two owned tiles
    // Loop tiles.  The dQ kernel keeps K and V in rings of their own: V_j is
    // free once dP_j is done, K_j only after dQ += dS_j K_j, and a third K
    // slot lets K_j+3 load while tile j+1 is worked on, so that no load waits
    // on the MMA that frees its slot.
    static constexpr int KSLOTS = 3, VSLOTS = 2;
    static constexpr int KRING = 2 * TILE_BYTES;
    static constexpr int VRING = KRING + KSLOTS * TILE_BYTES;
    // The dK/dV kernel works through each query tile in two halves of 64 rows
    // and keeps a ring of four half slots (Q rows, then dO rows, of one half)
    // with the half's row vectors (-LSE*log2e, then -D; 64 floats each): a
    // half's slot is free once that half's accumulation is done, a whole tile
    // period before the slot's next half is needed.
    static constexpr int HSLOTS = 4, HALF_BYTES = TILE_BYTES / 2, HPANEL = PANEL_BYTES / 2;
    static constexpr int HRING = 2 * TILE_BYTES;
    static constexpr int HVEC = HRING + HSLOTS * TILE_BYTES;
    static constexpr int HVEC_BYTES = 2 * (kT / 2) * 4;
    static constexpr int BARS = MODE_ == kDQ ? VRING + VSLOTS * TILE_BYTES : HVEC + HSLOTS * HVEC_BYTES;
    // at least 120 KB so that a second CTA never shares the SM: each
    // allocates all 512 TMEM columns; plus 1 KB to align for the swizzle
    static constexpr int SMEM_USED = BARS + 256;
    static constexpr int SMEM_BYTES = (SMEM_USED < 120 * 1024 ? 120 * 1024 : SMEM_USED) + 1024;
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
    // TMEM columns
    static constexpr int S_COL = 0, DP_COL = 128, ACC0 = 256, ACC1 = 256 + D;
    static constexpr int DS_COL = 384;                     // dQ kernel: dS of tile j at DS_COL + 64 * (j % 2)
    static_assert(ACC1 + D <= (int)kTmemCols, "TMEM budget");
    static_assert(DS_COL + 128 <= (int)kTmemCols, "dQ kernel: two 64-column dS buffers");
    static_assert(2 * HALF_BYTES == TILE_BYTES && 2 * HPANEL == PANEL_BYTES, "half slots split a tile in two");
};

struct BwdParams {
    const void *q, *k, *v, *o, *dout;   // q, o, dout [B, Sq, H, D]; k, v [B, Sk, H, D]
    const float *lse;                   // [B, H, Sq] natural-log LSE of the forward
    // workspace: per (b, h) row, sq_pad = Sq rounded up to 128 entries of
    // -LSE_i * log2(e) and -D_i (D_i = dO_i . O_i); -inf and 0 past Sq
    float *nl, *nd;
    int sq_pad;
    void *dq, *dk, *dv;
    int B, H, Sq, Sk;
    float scale, c2;                    // c2 = scale * log2(e)
    int mask, causal_type, off;         // off = Sk - Sq for a q-end causal mask, else 0
};

struct BwdBars {
    uint64_t own_full, own_empty, acc_full, drain;
    uint64_t acc_empty;                 // dK/dV: every compute warp has read the accumulators
    uint64_t turn[2];                   // dK/dV: issuing turn of lane a / lane b
    uint64_t s_full[2], c_full[2];      // dQ: index 0 only; dK/dV: one per half of the query tile
    uint64_t s_read;                    // dQ kernel: S and dP of the current tile are in registers
    uint64_t st_full[3], st_empty[3];   // dQ kernel: K slots
    uint64_t v_full[2], v_empty[2];     // dQ kernel: V slots
    uint64_t h_full[4], h_empty[4];     // dK/dV kernel: half slots
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(BwdBars) <= 256, "barrier block");

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

__device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, volatile int *abort_flag) {
    const unsigned long long t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63) == 0) {
            if (*abort_flag) return false;
            if (globaltimer() - t0 > g_bwd_wait_ns) {
                *abort_flag = 1;
                atomicExch(&g_bwd_status, FMHA_ERR_TIMEOUT);
                return false;
            }
        }
    }
}

// Bounded wait: the phase completes, the CTA aborts, or g_bwd_wait_ns pass.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    return mbar_wait_slow(bar, parity, abort_flag);
}

__device__ __noinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity) {
    const unsigned long long t0 = globaltimer();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer() - t0 > kDrainNs) return false;
    }
}

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag) {
    const bool r = mbar_wait(bar, parity, abort_flag);
    return __all_sync(0xffffffffu, r);
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *map, uint32_t bar, int c0, int c1,
                                            int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
        : "memory");
}

// Untiled bulk copy global -> shared (both 16-byte aligned, bytes a multiple
// of 16), completing on an mbarrier's transaction count.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
                 : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }


// Shared-memory descriptors as two 32-bit words.  The high word (stride
// byte offset, version, swizzle) is the same for every operand here; the low
// word holds the start address (16-byte units, 14 bits) and the leading byte
// offset, and adding (bytes >> 4) to it moves the start address only, since
// shared memory stays inside the 256 KB the field spans.  Each MMA then costs
// one 32-bit add for its k-step.
__host__ __device__ constexpr uint32_t desc_hi(uint32_t sbo, uint32_t swz) {
    return ((sbo >> 4) & 0x3FFFu) | (1u << 14) | (swz << 29);
}

__device__ __forceinline__ uint32_t desc_lo(uint32_t saddr, uint32_t lbo) {
    return ((saddr & 0x3FFFFu) >> 4) | (((lbo >> 4) & 0x3FFFu) << 16);
}



// MMA (D[tmem] (+)= A * B, A from shared memory or TMEM, B from shared memory),
// commit and arrive in warp-collective form: the whole (converged) warp
// executes them with warp-uniform operands and one elected lane issues the
// instruction, so the operand words can stay in uniform registers.
__device__ __forceinline__ void mma_ss_e(uint32_t d, uint32_t a_lo, uint32_t b_lo, uint32_t hi, uint32_t idesc,
                                         uint32_t acc) {
    asm volatile(
        "{\n.reg .pred p, e;\n.reg .b64 da, db;\nsetp.ne.b32 p, %4, 0;\nelect.sync _|e, 0xffffffff;\n"
        "mov.b64 da, {%1, %3};\nmov.b64 db, {%2, %3};\n"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, p;\n}\n" ::"r"(d),
        "r"(a_lo), "r"(b_lo), "r"(hi), "r"(acc), "r"(idesc)
        : "memory");
}

__device__ __forceinline__ void mma_ts_e(uint32_t d, uint32_t a, uint32_t b_lo, uint32_t hi, uint32_t idesc,
                                         uint32_t acc) {
    asm volatile(
        "{\n.reg .pred p, e;\n.reg .b64 db;\nsetp.ne.b32 p, %4, 0;\nelect.sync _|e, 0xffffffff;\n"
        "mov.b64 db, {%2, %3};\n"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], db, %5, p;\n}\n" ::"r"(d),
        "r"(a), "r"(b_lo), "r"(hi), "r"(acc), "r"(idesc)
        : "memory");
}

__device__ __forceinline__ void tc_commit_e(uint32_t bar) {
    asm volatile(
        "{\n.reg .pred e;\nelect.sync _|e, 0xffffffff;\n"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}\n" ::"r"(bar)
        : "memory");
}

__device__ __forceinline__ void mbar_arrive_e(uint32_t bar) {
    asm volatile(
        "{\n.reg .pred e;\nelect.sync _|e, 0xffffffff;\n"
        "@e mbarrier.arrive.shared::cta.b64 _, [%0];\n}\n" ::"r"(bar)
        : "memory");
}

__host__ __device__ constexpr uint32_t bwd_idesc(uint32_t fmt, int n, bool b_mn) {
    return (1u << 4) | (fmt << 7) | (fmt << 10) | ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(n >> 3) << 17) |
           ((uint32_t)(kT >> 4) << 24);
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

__device__ __forceinline__ void tmem_wait_ld2(uint32_t (&a)[32], uint32_t (&b)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3]), "+r"(a[4]), "+r"(a[5]), "+r"(a[6]), "+r"(a[7]),
                   "+r"(a[8]), "+r"(a[9]), "+r"(a[10]), "+r"(a[11]), "+r"(a[12]), "+r"(a[13]), "+r"(a[14]),
                   "+r"(a[15]), "+r"(a[16]), "+r"(a[17]), "+r"(a[18]), "+r"(a[19]), "+r"(a[20]), "+r"(a[21]),
                   "+r"(a[22]), "+r"(a[23]), "+r"(a[24]), "+r"(a[25]), "+r"(a[26]), "+r"(a[27]), "+r"(a[28]),
                   "+r"(a[29]), "+r"(a[30]), "+r"(a[31])
                 :
                 : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(b[0]), "+r"(b[1]), "+r"(b[2]), "+r"(b[3]), "+r"(b[4]), "+r"(b[5]), "+r"(b[6]), "+r"(b[7]),
                   "+r"(b[8]), "+r"(b[9]), "+r"(b[10]), "+r"(b[11]), "+r"(b[12]), "+r"(b[13]), "+r"(b[14]),
                   "+r"(b[15]), "+r"(b[16]), "+r"(b[17]), "+r"(b[18]), "+r"(b[19]), "+r"(b[20]), "+r"(b[21]),
                   "+r"(b[22]), "+r"(b[23]), "+r"(b[24]), "+r"(b[25]), "+r"(b[26]), "+r"(b[27]), "+r"(b[28]),
                   "+r"(b[29]), "+r"(b[30]), "+r"(b[31])
                 :
                 : "memory");
}

__device__ __forceinline__ void tmem_wait_ld1(uint32_t (&a)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3]), "+r"(a[4]), "+r"(a[5]), "+r"(a[6]), "+r"(a[7]),
                   "+r"(a[8]), "+r"(a[9]), "+r"(a[10]), "+r"(a[11]), "+r"(a[12]), "+r"(a[13]), "+r"(a[14]),
                   "+r"(a[15]), "+r"(a[16]), "+r"(a[17]), "+r"(a[18]), "+r"(a[19]), "+r"(a[20]), "+r"(a[21]),
                   "+r"(a[22]), "+r"(a[23]), "+r"(a[24]), "+r"(a[25]), "+r"(a[26]), "+r"(a[27]), "+r"(a[28]),
                   "+r"(a[29]), "+r"(a[30]), "+r"(a[31])
                 :
                 : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint64_t pack_f2(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}

__device__ __forceinline__ void unpack_f2(uint64_t v, float &a, float &b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}

// a * b + c on two fp32 lanes at once
__device__ __forceinline__ uint64_t fma_f2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

template <bool BF>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    uint32_t r;
    if constexpr (BF) asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    else asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

template <bool BF>
__device__ __forceinline__ float to_f32(uint16_t x) {
    if constexpr (BF) return __uint_as_float((uint32_t)x << 16);
    else return __half2float(__ushort_as_half(x));
}

// Is key kk visible to query qq (both inside the problem)?
__device__ __forceinline__ bool visible(const BwdParams &p, int qq, int kk) {
    return qq < p.Sq && kk < p.Sk && (p.mask != FMHA_MASK_CAUSAL || kk <= qq + p.off);
}

// ---------------------------------------------------------------------------
// Work units: (b, h, owned tile); the loop covers the tiles of the other side
// that hold a visible pair.
// ---------------------------------------------------------------------------

struct BUnit {
    int b, h, row0;                     // owned tile's first row (query row for dQ, key row for dK/dV)
    int j0, j1;                         // loop tiles [j0, j1)
};

template <int MODE>
__device__ __forceinline__ bool bwd_unit(const BwdParams &p, int u, BUnit &U) {
    const int own_tiles = MODE == kDQ ? (p.Sq + kT - 1) / kT : (p.Sk + kT - 1) / kT;
    const int per = p.B * p.H;
    if (u >= per * own_tiles) return false;
    const int r = u / per, rem = u - r * per;
    U.b = rem / p.H;
    U.h = rem - U.b * p.H;
    const bool causal = p.mask == FMHA_MASK_CAUSAL;
    if (MODE == kDQ) {
        // heaviest first: later query tiles see more keys under a causal mask
        const int t = causal ? own_tiles - 1 - r : r;
        U.row0 = t * kT;
        int nt, nu;
        kv_tile_range(U.row0, kT, p.Sq, p.Sk, p.mask, p.causal_type, kT, &nt, &nu);
        U.j0 = 0;
        U.j1 = nt;
    } else {
        // heaviest first: earlier key tiles are seen by more queries
        const int t = r;
        U.row0 = t * kT;
        const int q_tiles = (p.Sq + kT - 1) / kT;
        int first = 0;
        if (causal) {
            const int q_first = U.row0 - p.off;          // first query that sees key row0
            first = q_first <= 0 ? 0 : q_first / kT;
        }
        U.j0 = imin(first, q_tiles);
        U.j1 = (p.Sk > U.row0) ? q_tiles : U.j0;
    }
    return true;
}

// ---------------------------------------------------------------------------
// Roles
// ---------------------------------------------------------------------------

// Producer: the owned pair of tiles, then the loop tiles: K_j and V_j into
// their own rings for dQ; for dK/dV each query half (64 rows of Q_i and of
// dO_i, and the rows' -LSE * log2(e) and -D) into a half slot.  Every load
// is an asynchronous copy, so no thread of this warp waits on memory.
template <class C, int MODE>
__device__ void bwd_producer(const BwdParams &p, const CUtensorMap *tmQ, const CUtensorMap *tmK,
                             const CUtensorMap *tmV, const CUtensorMap *tmO, uint8_t *smem, BwdBars *bars,
                             int lane) {
    volatile int *abort_flag = &bars->abort;
    if (lane == 0) {
        prefetch_tmap(tmQ);
        prefetch_tmap(tmK);
        prefetch_tmap(tmV);
        prefetch_tmap(tmO);
    }
    // the owned tiles come from (Q, dO) for dQ and (K, V) for dK/dV; the loop
    // tiles from the other pair
    const CUtensorMap *own0 = MODE == kDQ ? tmQ : tmK, *own1 = MODE == kDQ ? tmO : tmV;
    const CUtensorMap *ld0 = MODE == kDQ ? tmK : tmQ, *ld1 = MODE == kDQ ? tmV : tmO;
    constexpr int KS = C::KSLOTS;
    uint32_t kfill = 0, vfill = 0, hfill = 0, owned = 0;   // loads issued into each ring
    bool ok = true;
    if (g_bwd_test_gate) {
        // a flag nothing sets: the wait runs out, records the timeout and
        // raises the abort flag; no copy has been issued yet
        const volatile int *flag = &g_bwd_test_flag;
        const unsigned long long t0 = globaltimer();
        for (uint32_t it = 1; !*flag; ++it) {
            if ((it & 63) == 0 && (*abort_flag || globaltimer() - t0 > g_bwd_wait_ns)) {
                *abort_flag = 1;
                atomicExch(&g_bwd_status, FMHA_ERR_TIMEOUT);
                break;
            }
        }
        ok = false;
    }
    for (int u = blockIdx.x; ok; u += gridDim.x) {
        BUnit U;
        if (!bwd_unit<MODE>(p, u, U)) break;
        if (U.j0 >= U.j1) continue;
        if (owned > 0 && !warp_wait(smem_u32(&bars->own_empty), (owned - 1) & 1, abort_flag)) {
            ok = false;
            break;
        }
        if (lane == 0) {
            const uint32_t fb = smem_u32(&bars->own_full);
            mbar_expect_tx(fb, 2 * C::TILE_BYTES);
#pragma unroll
            for (int pn = 0; pn < C::PANELS; ++pn) {
                tma_load_4d(smem_u32(smem + C::OWN + pn * C::PANEL_BYTES), own0, fb, pn * C::BOX_D, U.h, U.row0, U.b);
                tma_load_4d(smem_u32(smem + C::OWN + C::TILE_BYTES + pn * C::PANEL_BYTES), own1, fb, pn * C::BOX_D,
                            U.h, U.row0, U.b);
            }
        }
        ++owned;
        if constexpr (MODE == kDQ) {
            for (int j = U.j0; j < U.j1; ++j) {
                const int ks = kfill % KS;
                const uint32_t kr = kfill / KS;
                if (kr > 0 && !warp_wait(smem_u32(&bars->st_empty[ks]), (kr - 1) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                const uint32_t kb = smem_u32(&bars->st_full[ks]);
                const uint32_t kdst = smem_u32(smem + C::KRING + ks * C::TILE_BYTES);
                if (lane == 0) {
                    mbar_expect_tx(kb, C::TILE_BYTES);
#pragma unroll
                    for (int pn = 0; pn < C::PANELS; ++pn)
                        tma_load_4d(kdst + pn * C::PANEL_BYTES, ld0, kb, pn * C::BOX_D, U.h, j * kT, U.b);
                }
                ++kfill;
                const int vs = vfill & 1;
                const uint32_t vr = vfill >> 1;
                if (vr > 0 && !warp_wait(smem_u32(&bars->v_empty[vs]), (vr - 1) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                const uint32_t vb = smem_u32(&bars->v_full[vs]);
                const uint32_t vdst = smem_u32(smem + C::VRING + vs * C::TILE_BYTES);
                if (lane == 0) {
                    mbar_expect_tx(vb, C::TILE_BYTES);
#pragma unroll
                    for (int pn = 0; pn < C::PANELS; ++pn)
                        tma_load_4d(vdst + pn * C::PANEL_BYTES, ld1, vb, pn * C::BOX_D, U.h, j * kT, U.b);
                }
                ++vfill;
            }
        } else {
            // half x of loop tile j: 64 rows of Q and dO (64-row boxes) and the
            // rows' two vectors (bulk copies from the padded workspace rows)
            const int64_t vrow = ((int64_t)U.b * p.H + U.h) * p.sq_pad;
            for (int j = U.j0; j < U.j1 && ok; ++j) {
#pragma unroll 1
                for (int x = 0; x < 2; ++x) {
                    const int hs = hfill & 3;
                    const uint32_t hr = hfill >> 2;
                    if (hr > 0 && !warp_wait(smem_u32(&bars->h_empty[hs]), (hr - 1) & 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t hb = smem_u32(&bars->h_full[hs]);
                    const uint32_t dst = smem_u32(smem + C::HRING + hs * C::TILE_BYTES);
                    const uint32_t vdst = smem_u32(smem + C::HVEC + hs * C::HVEC_BYTES);
                    const int r0 = j * kT + x * (kT / 2);
                    if (lane == 0) {
                        mbar_expect_tx(hb, C::TILE_BYTES + C::HVEC_BYTES);
#pragma unroll
                        for (int pn = 0; pn < C::PANELS; ++pn) {
                            tma_load_4d(dst + pn * C::HPANEL, ld0, hb, pn * C::BOX_D, U.h, r0, U.b);
                            tma_load_4d(dst + C::HALF_BYTES + pn * C::HPANEL, ld1, hb, pn * C::BOX_D, U.h, r0, U.b);
                        }
                        bulk_load(vdst, p.nl + vrow + r0, C::HVEC_BYTES / 2, hb);
                        bulk_load(vdst + C::HVEC_BYTES / 2, p.nd + vrow + r0, C::HVEC_BYTES / 2, hb);
                    }
                    ++hfill;
                }
            }
        }
        if (!ok) break;
    }
    if (ok) {
        // the last releases of every slot and of the owned tiles
        if (MODE == kDQ) {
            for (int st = 0; st < KS; ++st) {
                const uint32_t nf = kfill > (uint32_t)st ? (kfill - st + KS - 1) / KS : 0;
                if (nf && !warp_wait(smem_u32(&bars->st_empty[st]), (nf - 1) & 1, abort_flag)) break;
            }
            for (int st = 0; st < 2; ++st) {
                const uint32_t nf = vfill > (uint32_t)st ? (vfill - st + 1) / 2 : 0;
                if (nf && !warp_wait(smem_u32(&bars->v_empty[st]), (nf - 1) & 1, abort_flag)) break;
            }
        } else {
            for (int st = 0; st < 4; ++st) {
                const uint32_t nf = hfill > (uint32_t)st ? (hfill - st + 3) / 4 : 0;
                if (nf && !warp_wait(smem_u32(&bars->h_empty[st]), (nf - 1) & 1, abort_flag)) break;
            }
        }
        if (owned) warp_wait(smem_u32(&bars->own_empty), (owned - 1) & 1, abort_flag);
    } else if (lane == 0) {
        // let the copies in flight land before the CTA exits
        for (uint32_t f = kfill > (uint32_t)KS ? kfill - KS : 0; f < kfill; ++f)
            mbar_wait_drain(smem_u32(&bars->st_full[f % KS]), (f / KS) & 1);
        for (uint32_t f = vfill > 2 ? vfill - 2 : 0; f < vfill; ++f)
            mbar_wait_drain(smem_u32(&bars->v_full[f & 1]), (f >> 1) & 1);
        for (uint32_t f = hfill > 4 ? hfill - 4 : 0; f < hfill; ++f)
            mbar_wait_drain(smem_u32(&bars->h_full[f & 3]), (f >> 2) & 1);
        if (owned) mbar_wait_drain(smem_u32(&bars->own_full), (owned - 1) & 1);
    }
}

// MMA issuer of the dQ kernel (warp kMmaWarp, converged; one elected lane
// issues each MMA, commit and arrive).  dS lives apart from S and dP (two
// buffers), so S and dP of tile j+1 are issued as soon as the compute warps
// have read S_j and dP_j (s_read), and dQ += dS_j K_j once dS_j is written
// (c_full): the elementwise work of tile j overlaps the MMAs of tile j+1.
// In issue order S_j+2 follows dQ_j, so "S_j+2 complete" implies "dS buffer
// j % 2 read".  V_j's slot is released after dP_j, K_j's after dQ_j.
template <class C, bool BF>
__device__ void bwd_mma_dq(const BwdParams &p, uint8_t *smem, BwdBars *bars, uint32_t tmem_any) {
    volatile int *abort_flag = &bars->abort;
    const uint32_t tmem = __shfl_sync(0xffffffffu, tmem_any, 0);   // the same in every lane
    constexpr uint32_t fmt = BF ? 1u : 0u;
    constexpr uint32_t kIdS = bwd_idesc(fmt, kT, false);
    constexpr uint32_t kIdAcc = bwd_idesc(fmt, C::D, true);
    constexpr int KS = C::KSLOTS;
    // descriptor words: K-major operands (LBO unused) and K read MN-major
    // (LBO = panel stride); each MMA adds its k-step's offset to the low word
    constexpr uint32_t kHi = desc_hi(C::SBO, (uint32_t)C::SW_CODE);
    constexpr uint32_t kTileStep = C::TILE_BYTES >> 4;
    const uint32_t a0 = desc_lo(smem_u32(smem + C::OWN), 16);                        // Q
    const uint32_t a1 = a0 + kTileStep;                                              // dO
    const uint32_t k_lo = desc_lo(smem_u32(smem + C::KRING), 16);
    const uint32_t kmn_lo = desc_lo(smem_u32(smem + C::KRING), C::PANEL_BYTES);
    const uint32_t v_lo = desc_lo(smem_u32(smem + C::VRING), 16);
    uint32_t cons = 0, owned = 0, cc = 0, rc = 0;
    bool ok = true;
    // S = Q K^T and dP = dO V^T of the loop tile with sequence number c
    auto issue_s = [&](uint32_t c) -> bool {
        const int ks = c % KS, vs = c & 1;
        if (!warp_wait(smem_u32(&bars->st_full[ks]), (c / KS) & 1, abort_flag)) return false;
        const uint32_t bk = k_lo + ks * kTileStep;
#pragma unroll
        for (int kk = 0; kk < C::D / 16; ++kk) {
            const uint32_t off = ((kk * 32 / C::SW) * C::PANEL_BYTES + (kk * 32) % C::SW) >> 4;
            mma_ss_e(tmem + C::S_COL, a0 + off, bk + off, kHi, kIdS, kk > 0 ? 1u : 0u);
        }
        if (!warp_wait(smem_u32(&bars->v_full[vs]), (c >> 1) & 1, abort_flag)) return false;
        const uint32_t bv = v_lo + vs * kTileStep;
#pragma unroll
        for (int kk = 0; kk < C::D / 16; ++kk) {
            const uint32_t off = ((kk * 32 / C::SW) * C::PANEL_BYTES + (kk * 32) % C::SW) >> 4;
            mma_ss_e(tmem + C::DP_COL, a1 + off, bv + off, kHi, kIdS, kk > 0 ? 1u : 0u);
        }
        tc_commit_e(smem_u32(&bars->v_empty[vs]));
        return true;
    };
    for (int u = blockIdx.x; ok; u += gridDim.x) {
        BUnit U;
        if (!bwd_unit<kDQ>(p, u, U)) break;
        if (U.j0 >= U.j1) continue;
        if (!warp_wait(smem_u32(&bars->own_full), owned & 1, abort_flag)) break;
        ++owned;
        uint32_t cur = cons;                 // sequence number of tile j
        if (!issue_s(cons++)) break;
        if (U.j0 + 1 == U.j1) tc_commit_e(smem_u32(&bars->own_empty));
        tc_commit_e(smem_u32(&bars->s_full[0]));
        for (int j = U.j0; j < U.j1; ++j) {
            if (!warp_wait(smem_u32(&bars->s_read), rc & 1, abort_flag)) { ok = false; break; }
            ++rc;
            if (j + 1 < U.j1) {
                tc_fence_after();
                if (!issue_s(cons++)) { ok = false; break; }
                if (j + 2 == U.j1) tc_commit_e(smem_u32(&bars->own_empty));
                tc_commit_e(smem_u32(&bars->s_full[0]));
            }
            if (!warp_wait(smem_u32(&bars->c_full[0]), cc & 1, abort_flag)) { ok = false; break; }
            ++cc;
            tc_fence_after();
            // dQ += dS_j K_j: A = dS buffer j % 2 (16-bit, 8 columns per step of
            // 16 keys), B = K_j rows MN-major
            const int ks = cur % KS;
            const uint32_t ds = tmem + C::DS_COL + 64 * (j & 1);
            const uint32_t bk = kmn_lo + ks * kTileStep;
#pragma unroll
            for (int kk = 0; kk < kT / 16; ++kk)
                mma_ts_e(tmem + C::ACC0, ds + kk * 8, bk + ((kk * 16 * C::SW) >> 4), kHi, kIdAcc,
                         (j > U.j0 || kk > 0) ? 1u : 0u);
            tc_commit_e(smem_u32(&bars->st_empty[ks]));
            ++cur;
        }
        if (!ok) break;
        tc_commit_e(smem_u32(&bars->acc_full));
    }
    tc_commit_e(smem_u32(&bars->drain));
    mbar_wait_drain(smem_u32(&bars->drain), 0);
}

// MMA issuers of the dK/dV kernel: warp kMmaWarp for query half a, warp
// kMmaWarp2 for half b; the whole warp runs the loop with warp-uniform values
// and one elected lane issues each MMA, commit and arrive.  The loop tile's
// 128 queries are taken in two halves of 64 with TMEM of their own: S^T and
// dP^T of half x (M = 128 keys, N = 64 queries) land in columns S_COL + 64x
// and DP_COL + 64x, the compute warps turn them into P^T and dS^T in place,
// and dV += P^T dO, dK += dS^T Q then take the half's 64 queries as the
// reduction.  While one half is in the compute warps the MMAs of the other
// run, so the tensor pipe and the elementwise work overlap.
//
// The two warps take turns; turn k of warp x issues acc(x, i-1) and
// S/dP(x, i) for loop tile i = j0 + k (the first turn of a unit has no
// accumulation, the last no S/dP), so the pipe sees a, b, a, b, ... and "S^T
// of half x of tile i complete" implies "the accumulation from half x of tile
// i-1 complete", which is what lets S^T overwrite P^T.  A warp does its waits
// (c_full, the half slot, the previous unit's epilogue) before taking its
// turn, while the other warp issues, and hands the turn over two MMAs before
// its last one, so the pipe never drains between turns: an MMA holds its
// issuing thread for most of its pipe time, and one issuer alone cannot both
// issue and wait.  Warp a's first accumulation of a unit overwrites dV and dK;
// warp b's comes a turn later.
template <class C, bool BF>
__device__ void bwd_mma_dkdv(const BwdParams &p, uint8_t *smem, BwdBars *bars, uint32_t tmem_any, int x) {
    volatile int *abort_flag = &bars->abort;
    const uint32_t tmem = __shfl_sync(0xffffffffu, tmem_any, 0);   // the same in every lane
    constexpr uint32_t fmt = BF ? 1u : 0u;
    constexpr uint32_t kIdS = bwd_idesc(fmt, kT / 2, false);
    constexpr uint32_t kIdAcc = bwd_idesc(fmt, C::D, true);
    constexpr int kSteps = C::D / 16;                  // MMAs of one S^T (or dP^T)
    constexpr int kPassAt = 2 * kSteps - 3;            // S/dP MMA (index) after which the turn passes
    static_assert(kPassAt >= 0 && kPassAt < 2 * kSteps, "the turn passes exactly once per S/dP group");
    // descriptor words (see bwd_mma_dq); half slot hs starts hs tiles into the ring
    constexpr uint32_t kHi = desc_hi(C::SBO, (uint32_t)C::SW_CODE);
    constexpr uint32_t kTileStep = C::TILE_BYTES >> 4, kHalfStep = C::HALF_BYTES >> 4;
    const uint32_t a0 = desc_lo(smem_u32(smem + C::OWN), 16);                        // K (owned)
    const uint32_t a1 = a0 + kTileStep;                                              // V (owned)
    const uint32_t h_lo = desc_lo(smem_u32(smem + C::HRING), 16);
    const uint32_t hmn_lo = desc_lo(smem_u32(smem + C::HRING), C::HPANEL);
    const uint32_t my_turn = smem_u32(&bars->turn[x]), next_turn = smem_u32(&bars->turn[x ^ 1]);
    uint32_t cons = 0, owned = 0, cc = 0, units = 0, turns = 0;
    bool ok = true;
    // S^T and dP^T of half x from half slot hs (B = its 64 rows of Q_i, dO_i);
    // passes the turn two MMAs before the end
    auto issue_sdp = [&](int hs) {
        const uint32_t bq = h_lo + hs * kTileStep, bo = bq + kHalfStep;
        const uint32_t ds = tmem + C::S_COL + 64 * x, dd = tmem + C::DP_COL + 64 * x;
#pragma unroll
        for (int kk = 0; kk < kSteps; ++kk) {
            const uint32_t oa = ((kk * 32 / C::SW) * C::PANEL_BYTES + (kk * 32) % C::SW) >> 4;
            const uint32_t ob = ((kk * 32 / C::SW) * C::HPANEL + (kk * 32) % C::SW) >> 4;
            mma_ss_e(ds, a0 + oa, bq + ob, kHi, kIdS, kk > 0 ? 1u : 0u);
            if (kk == kPassAt) mbar_arrive_e(next_turn);
        }
#pragma unroll
        for (int kk = 0; kk < kSteps; ++kk) {
            const uint32_t oa = ((kk * 32 / C::SW) * C::PANEL_BYTES + (kk * 32) % C::SW) >> 4;
            const uint32_t ob = ((kk * 32 / C::SW) * C::HPANEL + (kk * 32) % C::SW) >> 4;
            mma_ss_e(dd, a1 + oa, bo + ob, kHi, kIdS, kk > 0 ? 1u : 0u);
            if (kSteps + kk == kPassAt) mbar_arrive_e(next_turn);
        }
        tc_commit_e(smem_u32(&bars->s_full[x]));
    };
    // dV += P^T_x dO_x and dK += dS^T_x Q_x over the half's 64 queries (16 per
    // MMA): A = 16-bit values in TMEM (8 columns per step), B = the slot's
    // rows MN-major
    auto issue_acc = [&](int hs, bool first) {
        const uint32_t bq = hmn_lo + hs * kTileStep, bo = bq + kHalfStep;
        const uint32_t ps = tmem + C::S_COL + 64 * x, pd = tmem + C::DP_COL + 64 * x;
        // queries 0-31 of the half are packed in columns 0-15, queries 32-63
        // in columns 32-47 (each compute warp writes over its own columns)
#pragma unroll
        for (int kk = 0; kk < kT / 32; ++kk)
            mma_ts_e(tmem + C::ACC0, ps + (kk >> 1) * 32 + (kk & 1) * 8, bo + ((kk * 16 * C::SW) >> 4), kHi, kIdAcc,
                     (!first || kk > 0) ? 1u : 0u);                 // dV
#pragma unroll
        for (int kk = 0; kk < kT / 32; ++kk)
            mma_ts_e(tmem + C::ACC1, pd + (kk >> 1) * 32 + (kk & 1) * 8, bq + ((kk * 16 * C::SW) >> 4), kHi, kIdAcc,
                     (!first || kk > 0) ? 1u : 0u);                 // dK
    };
    // half slot and its fill phase of half x of the loop tile with sequence number c
    auto slot = [&](uint32_t c) { return (int)((2 * c + x) & 3); };
    auto slot_phase = [&](uint32_t c) { return ((2 * c + x) >> 2) & 1; };
    for (int u = blockIdx.x; ok; u += gridDim.x) {
        BUnit U;
        if (!bwd_unit<kDKDV>(p, u, U)) break;
        if (U.j0 >= U.j1) continue;
        const int n = U.j1 - U.j0;
        for (int k = 0; k <= n; ++k) {
            // waits first, while the other lane holds the turn
            bool w = true;
            if (k == 0) w = warp_wait(smem_u32(&bars->own_full), owned & 1, abort_flag);
            if (w && k > 0) w = warp_wait(smem_u32(&bars->c_full[x]), cc & 1, abort_flag);
            if (w && k == 1 && x == 0 && units > 0)
                w = warp_wait(smem_u32(&bars->acc_empty), (units - 1) & 1, abort_flag);
            if (w && k < n) w = warp_wait(smem_u32(&bars->h_full[slot(cons + k)]), slot_phase(cons + k), abort_flag);
            if (w) w = warp_wait(my_turn, turns & 1, abort_flag);
            if (!w) {
                ok = false;
                break;
            }
            ++turns;
            tc_fence_after();
            if (k > 0) {
                ++cc;
                const int hs = slot(cons + k - 1);
                issue_acc(hs, k == 1 && x == 0);
                tc_commit_e(smem_u32(&bars->h_empty[hs]));    // the half slot is read
            }
            if (k < n) {
                issue_sdp(slot(cons + k));
                if (k == n - 1) tc_commit_e(smem_u32(&bars->own_empty));
            } else {
                mbar_arrive_e(next_turn);
            }
        }
        if (!ok) break;
        ++owned;
        cons += n;
        tc_commit_e(smem_u32(&bars->acc_full));
        ++units;
    }
    tc_commit_e(smem_u32(&bars->drain));
    mbar_wait_drain(smem_u32(&bars->drain), 0);
}

// Store 32 fp32 accumulator columns times mul as 16-bit values (64 bytes).
template <bool BF>
__device__ __forceinline__ void store32(uint8_t *dst, const uint32_t (&r)[32], float mul) {
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) w[i] = pack2<BF>(__uint_as_float(r[2 * i]) * mul, __uint_as_float(r[2 * i + 1]) * mul);
    uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
    for (int i = 0; i < 4; ++i) d4[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
}

// One 32-column chunk of the elementwise work for this thread's row:
// P = exp2(S * scale * log2e - LSE * log2e) (zero where masked) and
// dS = P (dP - D), from the chunk's S and dP values; packed to 16-bit pairs.
// nl / nd are -LSE*log2e and -D: per row in the dQ kernel, per column (read
// from the half slot's vectors, four at a time) in the dK/dV kernel.  FULL: every
// pair of the tile is visible, no per-element test.
template <bool BF, int MODE, bool FULL>
__device__ __forceinline__ void bwd_chunk(const BwdParams &p, const uint32_t (&s)[32], const uint32_t (&dp)[32],
                                          uint64_t c2x2, uint64_t nl_row, uint64_t nd_row, const float *vec_l,
                                          const float *vec_d, int row, int col0, uint32_t (&pw)[16],
                                          uint32_t (&dw)[16]) {
    const uint64_t ones = pack_f2(1.f, 1.f), zero2 = pack_f2(0.f, 0.f);
#pragma unroll
    for (int e = 0; e < 32; e += 4) {
        uint64_t nl[2] = {nl_row, nl_row}, nd[2] = {nd_row, nd_row};
        if constexpr (MODE == kDKDV) {
            const float4 lv = *reinterpret_cast<const float4 *>(vec_l + e);
            const float4 dv = *reinterpret_cast<const float4 *>(vec_d + e);
            nl[0] = pack_f2(lv.x, lv.y);
            nl[1] = pack_f2(lv.z, lv.w);
            nd[0] = pack_f2(dv.x, dv.y);
            nd[1] = pack_f2(dv.z, dv.w);
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int x = e + 2 * h;
            float a, b;
            unpack_f2(fma_f2(pack_f2(__uint_as_float(s[x]), __uint_as_float(s[x + 1])), c2x2, nl[h]), a, b);
            a = ex2(a);
            b = ex2(b);
            if constexpr (!FULL) {
                const int col = col0 + x;
                const bool va = MODE == kDQ ? visible(p, row, col) : visible(p, col, row);
                const bool vb = MODE == kDQ ? visible(p, row, col + 1) : visible(p, col + 1, row);
                a = va ? a : 0.f;
                b = vb ? b : 0.f;
            }
            const uint64_t diff = fma_f2(pack_f2(__uint_as_float(dp[x]), __uint_as_float(dp[x + 1])), ones, nd[h]);
            float da, db;
            unpack_f2(fma_f2(pack_f2(a, b), diff, zero2), da, db);
            pw[x / 2] = pack2<BF>(a, b);
            dw[x / 2] = pack2<BF>(da, db);
        }
    }
}

template <bool BF, int MODE>
__device__ __forceinline__ void bwd_chunk_sel(bool full, const BwdParams &p, const uint32_t (&s)[32],
                                              const uint32_t (&dp)[32], uint64_t c2x2, uint64_t nl_row,
                                              uint64_t nd_row, const float *vec_l, const float *vec_d, int row,
                                              int col0, uint32_t (&pw)[16], uint32_t (&dw)[16]) {
    if (full) bwd_chunk<BF, MODE, true>(p, s, dp, c2x2, nl_row, nd_row, vec_l, vec_d, row, col0, pw, dw);
    else bwd_chunk<BF, MODE, false>(p, s, dp, c2x2, nl_row, nd_row, vec_l, vec_d, row, col0, pw, dw);
}

// Elementwise work and epilogue: warps w and w+4 share TMEM lanes
// 32*(w%4)..+31 (rows of the owned tile).  dQ kernel: they take the lower /
// upper 64 columns of every loop tile.  dK/dV kernel: they take the lower /
// upper 32 columns of each query half, half a then half b, as soon as that
// half's S^T and dP^T are in TMEM.  In the epilogue, the lower / upper half
// of the head dimension.
template <class C, bool BF, int MODE>
__device__ void bwd_compute(const BwdParams &p, uint8_t *smem, BwdBars *bars, uint32_t tmem, int warp, int lane) {
    volatile int *abort_flag = &bars->abort;
    const int half = warp >> 2, wq = warp & 3;
    const int t = wq * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(wq * 32) << 16);
    const uint64_t c2x2 = pack_f2(p.c2, p.c2);
    uint32_t sph = 0, aph = 0, cons = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok; u += gridDim.x) {
        BUnit U;
        if (!bwd_unit<MODE>(p, u, U)) break;
        const int row = U.row0 + t;
        const bool have = U.j0 < U.j1;
        uint64_t nl_row = 0, nd_row = 0;
        int nu = 0;                                   // dQ: leading key tiles visible to every row
        if (MODE == kDQ) {
            // a row past Sq reads the padding (-inf, 0): P = 0
            const int64_t li = ((int64_t)U.b * p.H + U.h) * p.sq_pad + row;
            const float nl = p.nl[li], nd = p.nd[li];
            nl_row = pack_f2(nl, nl);
            nd_row = pack_f2(nd, nd);
            int nt;
            kv_tile_range(U.row0, kT, p.Sq, p.Sk, p.mask, p.causal_type, kT, &nt, &nu);
        }
        if constexpr (MODE == kDQ) {
            for (int j = U.j0; j < U.j1 && ok; ++j) {
                const bool got = warp_wait(smem_u32(&bars->s_full[0]), sph, abort_flag);
                sph ^= 1;
                if (!got) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // every (query, key) pair of the tile visible: no per-element
                // mask (rows and columns outside the problem already give P = 0
                // or touch only discarded rows)
                const bool full = j < nu;
                // S and dP of this warp's 64 columns, two chunks of 32
                const uint32_t sc = lane_base + C::S_COL + 64 * half, dc = lane_base + C::DP_COL + 64 * half;
                uint32_t s0[32], d0[32], s1[32], d1[32];
                tmem_ld32(sc, s0);
                tmem_ld32(dc, d0);
                tmem_wait_ld2(s0, d0);
                tmem_ld32(sc + 32, s1);
                tmem_ld32(dc + 32, d1);
                tmem_wait_ld2(s1, d1);
                const int col0 = j * kT + 64 * half;
                // S and dP may now be overwritten by the next tile's MMAs
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&bars->s_read));
                const uint32_t ds = lane_base + C::DS_COL + 64 * (j & 1) + 32 * half;
                {
                    uint32_t pw[16], dw[16];
                    bwd_chunk_sel<BF, MODE>(full, p, s0, d0, c2x2, nl_row, nd_row, nullptr, nullptr, row, col0, pw, dw);
                    tmem_st16(ds, dw);
                }
                {
                    uint32_t pw[16], dw[16];
                    bwd_chunk_sel<BF, MODE>(full, p, s1, d1, c2x2, nl_row, nd_row, nullptr, nullptr, row, col0 + 32, pw, dw);
                    tmem_st16(ds + 16, dw);
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&bars->c_full[0]));
            }
        } else {
            // every warp takes both query halves of a tile in turn, 32 of the
            // half's 64 columns each (c32); P^T and dS^T of those 32 queries go
            // back, as 16-bit pairs, over the first 16 of this warp's own 32
            // columns of S^T and dP^T, which no other warp reads
            const int c32 = 32 * half;
            for (int j = U.j0; j < U.j1 && ok; ++j) {
#pragma unroll 1
                for (int x = 0; x < 2; ++x) {
                    const int hs = (int)((2 * cons + x) & 3);          // the half's slot
                    const uint32_t hph = ((2 * cons + x) >> 2) & 1;
                    bool got = warp_wait(smem_u32(&bars->s_full[x]), (sph >> x) & 1, abort_flag);
                    sph ^= 1u << x;
                    // the slot's row vectors, written by the producer warp
                    if (got) got = warp_wait(smem_u32(&bars->h_full[hs]), hph, abort_flag);
                    if (!got) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const int col0 = j * kT + 64 * x + c32;
                    const bool full = p.mask != FMHA_MASK_CAUSAL || col0 + p.off >= U.row0 + kT - 1;
                    const uint32_t sc = lane_base + C::S_COL + 64 * x + c32, dc = lane_base + C::DP_COL + 64 * x + c32;
                    uint32_t s0[32], d0[32];
                    tmem_ld32(sc, s0);
                    tmem_ld32(dc, d0);
                    tmem_wait_ld2(s0, d0);
                    const float *vec = reinterpret_cast<const float *>(smem + C::HVEC + hs * C::HVEC_BYTES) + c32;
                    uint32_t pw[16], dw[16];
                    bwd_chunk_sel<BF, MODE>(full, p, s0, d0, c2x2, 0, 0, vec, vec + kT / 2, row, col0, pw, dw);
                    tmem_st16(sc, pw);
                    tmem_st16(dc, dw);
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&bars->c_full[x]));
                }
                ++cons;
            }
        }
        if (!ok) break;
        // epilogue: this warp's half of the head dimension.  The TMEM loads are
        // warp-wide (.sync.aligned): every lane takes part, whether or not its
        // row exists; only the stores are per row.
        if (have) {
            if (!warp_wait(smem_u32(&bars->acc_full), aph, abort_flag)) break;
            aph ^= 1;
            tc_fence_after();
        }
        constexpr int HC = C::D / 64;                 // 32-column chunks per half
        if (MODE == kDQ) {
            const bool keep = row < p.Sq;
            uint8_t *dst = static_cast<uint8_t *>(p.dq) + (((int64_t)U.b * p.Sq + row) * p.H + U.h) * C::ROW;
#pragma unroll 1
            for (int cc = 0; cc < HC; ++cc) {
                const int c = half * HC + cc;
                uint32_t r[32];
                if (have) {
                    tmem_ld32(lane_base + C::ACC0 + 32 * c, r);
                    tmem_wait_ld1(r);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) r[i] = 0u;
                }
                if (keep) store32<BF>(dst + c * 64, r, p.scale);
            }
        } else {
            const bool keep = row < p.Sk;
            const int64_t ro = (((int64_t)U.b * p.Sk + row) * p.H + U.h) * C::ROW;
            uint8_t *dvd = static_cast<uint8_t *>(p.dv) + ro;
            uint8_t *dkd = static_cast<uint8_t *>(p.dk) + ro;
#pragma unroll 1
            for (int cc = 0; cc < HC; ++cc) {
                const int c = half * HC + cc;
                uint32_t rv[32], rk[32];
                if (have) {
                    tmem_ld32(lane_base + C::ACC0 + 32 * c, rv);
                    tmem_ld32(lane_base + C::ACC1 + 32 * c, rk);
                    tmem_wait_ld2(rv, rk);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) rv[i] = rk[i] = 0u;
                }
                if (keep) {
                    store32<BF>(dvd + c * 64, rv, 1.f);
                    store32<BF>(dkd + c * 64, rk, p.scale);
                }
            }
            if (have) {
                // the accumulators may now be overwritten by the next unit
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&bars->acc_empty));
            }
        }
    }
}

template <class C, bool BF, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    fmha_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                    const BwdParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    BwdBars *bars = reinterpret_cast<BwdBars *>(smem + C::BARS);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        // dK/dV: both issuing warps commit the owned-tile, accumulator and
        // drain barriers
        const uint32_t issuers = MODE == kDKDV ? 2 : 1;
        mbar_init(smem_u32(&bars->own_full), 1);
        mbar_init(smem_u32(&bars->own_empty), issuers);
        for (int x = 0; x < 2; ++x) {
            mbar_init(smem_u32(&bars->s_full[x]), 1);
            // every compute warp arrives (dQ uses index 0 only)
            mbar_init(smem_u32(&bars->c_full[x]), kCompWarps);
        }
        mbar_init(smem_u32(&bars->s_read), kCompWarps);
        mbar_init(smem_u32(&bars->acc_full), issuers);
        mbar_init(smem_u32(&bars->drain), issuers);
        mbar_init(smem_u32(&bars->turn[0]), 1);
        mbar_init(smem_u32(&bars->turn[1]), 1);
        mbar_init(smem_u32(&bars->acc_empty), kCompWarps);
        for (int s = 0; s < 3; ++s) {
            mbar_init(smem_u32(&bars->st_full[s]), 1);
            mbar_init(smem_u32(&bars->st_empty[s]), 1);
        }
        for (int s = 0; s < 4; ++s) {
            // the copies' transaction count; freed by the issuing warp of its half
            mbar_init(smem_u32(&bars->h_full[s]), 1);
            mbar_init(smem_u32(&bars->h_empty[s]), 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(smem_u32(&bars->v_full[s]), 1);
            mbar_init(smem_u32(&bars->v_empty[s]), 1);
        }
        bars->abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        mbar_arrive(smem_u32(&bars->turn[0]));          // lane a issues first
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(&bars->tmem_base), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    if (warp < kCompWarps) {
        bwd_compute<C, BF, MODE>(p, smem, bars, tmem, warp, lane);
    } else if (warp == kProdWarp) {
        bwd_producer<C, MODE>(p, &tmQ, &tmK, &tmV, &tmO, smem, bars, lane);
    } else {
        if constexpr (MODE == kDQ) {
            if (warp == kMmaWarp) bwd_mma_dq<C, BF>(p, smem, bars, tmem);
        } else {
            bwd_mma_dkdv<C, BF>(p, smem, bars, tmem, warp == kMmaWarp ? 0 : 1);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) {
        __syncwarp();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// D_i = dO_i . O_i in fp32, one warp per (b, i, h) row with i < sq_pad; the
// row's workspace entries -LSE_i * log2(e) and -D_i (padding: -inf and 0).
template <int D, bool BF>
__global__ void fmha_bwd_dot_kernel(const BwdParams p) {
    const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    const int64_t rows = (int64_t)p.B * p.sq_pad * p.H;
    if (row >= rows) return;
    const int64_t h = row % p.H, bi = row / p.H, i = bi % p.sq_pad, b = bi / p.sq_pad;
    const int64_t w = (b * p.H + h) * p.sq_pad + i;
    if (i >= p.Sq) {
        if (lane == 0) {
            p.nl[w] = -INFINITY;
            p.nd[w] = 0.f;
        }
        return;
    }
    const int64_t src = (b * p.Sq + i) * p.H + h;
    const uint16_t *o = static_cast<const uint16_t *>(p.o) + src * D;
    const uint16_t *g = static_cast<const uint16_t *>(p.dout) + src * D;
    float acc = 0.f;
#pragma unroll
    for (int d = lane; d < D; d += 32) acc += to_f32<BF>(o[d]) * to_f32<BF>(g[d]);
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
    if (lane == 0) {
        p.nl[w] = -p.lse[(b * p.H + h) * p.Sq + i] * kLog2e;
        p.nd[w] = -acc;
    }
}

PFN_cuTensorMapEncodeTiled_v12000 bwd_encode_fn() {
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

int bwd_sm_count() {
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

// [B, rows, H, D] with a box of one head, 128 rows and one swizzle panel.
template <class C>
bool bwd_map(CUtensorMap *m, const void *base, bool bf, int H, int rows, int B, int box_rows = kT) {
    auto fn = bwd_encode_fn();
    if (!fn) return false;
    cuuint64_t dims[4] = {(cuuint64_t)C::D, (cuuint64_t)H, (cuuint64_t)(rows > 0 ? rows : 1), (cuuint64_t)B};
    cuuint64_t strides[3] = {(cuuint64_t)C::ROW, (cuuint64_t)C::ROW * H, (cuuint64_t)C::ROW * H * (rows > 0 ? rows : 1)};
    cuuint32_t box[4] = {(cuuint32_t)C::BOX_D, 1, (cuuint32_t)box_rows, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return fn(m, bf ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, const_cast<void *>(base),
              dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
              C::SW == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <class C, int MODE>
int bwd_launch_mode(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv, const CUtensorMap &to,
                    const BwdParams &p, bool bf, int sms, cudaStream_t stream) {
    const int own = MODE == kDQ ? (p.Sq + kT - 1) / kT : (p.Sk + kT - 1) / kT;
    const int64_t units = (int64_t)p.B * p.H * own;
    const int grid = (int)(units < sms ? units : sms);
    if (grid <= 0) return FMHA_OK;
    auto kern = bf ? fmha_bwd_kernel<C, true, MODE> : fmha_bwd_kernel<C, false, MODE>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES) != cudaSuccess)
        return FMHA_ERR_CUDA;
    kern<<<grid, kThreads, C::SMEM_BYTES, stream>>>(tq, tk, tv, to, p);
    return cudaGetLastError() == cudaSuccess ? FMHA_OK : FMHA_ERR_CUDA;
}

template <int D>
int bwd_launch(const BwdParams &p, bool bf, cudaStream_t stream) {
    using C = BCfg<D, kDQ>;
    CUtensorMap tq, tk, tv, to;
    if (!bwd_map<C>(&tq, p.q, bf, p.H, p.Sq, p.B) || !bwd_map<C>(&tk, p.k, bf, p.H, p.Sk, p.B) ||
        !bwd_map<C>(&tv, p.v, bf, p.H, p.Sk, p.B) || !bwd_map<C>(&to, p.dout, bf, p.H, p.Sq, p.B))
        return FMHA_ERR_CUDA;
    const int sms = bwd_sm_count();
    if (sms <= 0) return FMHA_ERR_CUDA;
    // 1) D_i = dO_i . O_i
    const int64_t rows = (int64_t)p.B * p.sq_pad * p.H;
    auto dot = bf ? fmha_bwd_dot_kernel<D, true> : fmha_bwd_dot_kernel<D, false>;
    dot<<<(unsigned)((rows + 7) / 8), 256, 0, stream>>>(p);
    if (cudaGetLastError() != cudaSuccess) return FMHA_ERR_CUDA;
    // 2) dQ, 3) dK and dV; the dK/dV kernel loads Q and dO in halves of 64 rows
    const int r = bwd_launch_mode<BCfg<D, kDQ>, kDQ>(tq, tk, tv, to, p, bf, sms, stream);
    if (r != FMHA_OK) return r;
    CUtensorMap tq2, to2;
    if (!bwd_map<C>(&tq2, p.q, bf, p.H, p.Sq, p.B, kT / 2) || !bwd_map<C>(&to2, p.dout, bf, p.H, p.Sq, p.B, kT / 2))
        return FMHA_ERR_CUDA;
    return bwd_launch_mode<BCfg<D, kDKDV>, kDKDV>(tq2, tk, tv, to2, p, bf, sms, stream);
}

// e4m3 inputs: every e4m3 value is a bf16 value, so the inputs are widened
// exactly into the workspace and differentiated on the bf16 path.  One launch
// for the five tensors; each thread converts 16 codes (16 bytes in, 32 out).
struct Widen {
    const uint8_t *src[5];
    __nv_bfloat16 *dst[5];
    int64_t n16[5];                     // 16-element groups of each tensor (its size is a multiple of 64)
};

__global__ void __launch_bounds__(256) widen_e4m3_kernel(const Widen w) {
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int t = 0; t < 5; ++t) {
        for (int64_t g = i; g < w.n16[t]; g += stride) {
            const uint4 x = reinterpret_cast<const uint4 *>(w.src[t])[g];
            const uint32_t in[4] = {x.x, x.y, x.z, x.w};
            uint32_t out[8];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const __nv_fp8x2_storage_t two = (__nv_fp8x2_storage_t)(in[k] >> (16 * h));
                    const float2 f = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(two, __NV_E4M3)));
                    const __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);
                    out[2 * k + h] = *reinterpret_cast<const uint32_t *>(&b);
                }
            }
            uint4 *d = reinterpret_cast<uint4 *>(w.dst[t]) + 2 * g;
            d[0] = make_uint4(out[0], out[1], out[2], out[3]);
            d[1] = make_uint4(out[4], out[5], out[6], out[7]);
        }
    }
}

}  // namespace

int bwd_set_wait_limit(unsigned long long ns) {
    const unsigned long long v = ns ? ns : kTimeoutNs;
    if (cudaMemcpyToSymbol(g_bwd_wait_ns, &v, sizeof(v)) != cudaSuccess) {
        cudaGetLastError();
        return FMHA_ERR_CUDA;
    }
    return FMHA_OK;
}

int bwd_set_test_gate(int on) {
    const int v = on ? 1 : 0;
    if (cudaMemcpyToSymbol(g_bwd_test_gate, &v, sizeof(v)) != cudaSuccess) {
        cudaGetLastError();
        return FMHA_ERR_CUDA;
    }
    return FMHA_OK;
}

int bwd_read_status(int reset) {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_bwd_status, sizeof(int)) != cudaSuccess) return FMHA_ERR_CUDA;
    if (reset && v != 0) {
        const int z = 0;
        if (cudaMemcpyToSymbol(g_bwd_status, &z, sizeof(int)) != cudaSuccess) return FMHA_ERR_CUDA;
    }
    return v;
}

}  // namespace fmha

using namespace fmha;

// Two fp32 vectors per (b, h) row of Sq rounded up to 128 entries.
extern "C" size_t fmha_bwd_workspace_size(int B, int H, int Sq) {
    if (B <= 0 || H <= 0 || Sq <= 0) return 0;
    const size_t sq_pad = ((size_t)Sq + kT - 1) / kT * kT;
    return 2 * (size_t)B * H * sq_pad * sizeof(float);
}

namespace {
// e4m3 workspace: the row vectors, then bf16 copies of q, o, dout (B*Sq*H*D
// each) and k, v (B*Sk*H*D each), every region 256-byte aligned.
size_t align256(size_t x) { return (x + 255) / 256 * 256; }
struct WidenLayout {
    size_t q, o, dout, k, v, total;
};
WidenLayout widen_layout(int B, int H, int Sq, int Sk, int D) {
    WidenLayout l;
    const size_t qb = (size_t)B * Sq * H * D * 2, kb = (size_t)B * Sk * H * D * 2;
    l.q = align256(fmha_bwd_workspace_size(B, H, Sq));
    l.o = l.q + align256(qb);
    l.dout = l.o + align256(qb);
    l.k = l.dout + align256(qb);
    l.v = l.k + align256(kb);
    l.total = l.v + kb;
    return l;
}
}  // namespace

extern "C" size_t fmha_bwd_workspace_size_ex(int B, int H, int Sq, int Sk, int D, int dtype) {
    if (B <= 0 || H <= 0 || Sq <= 0 || Sk < 0 || (D != 64 && D != 128)) return 0;
    if (dtype == FMHA_F16 || dtype == FMHA_BF16) return fmha_bwd_workspace_size(B, H, Sq);
    if (dtype != FMHA_E4M3) return 0;
    return widen_layout(B, H, Sq, Sk, D).total;
}

extern "C" int fmha_bwd(fmha_tensor q, fmha_tensor k, fmha_tensor v, fmha_tensor o, fmha_tensor dout,
                        const float *lse, fmha_tensor dq, fmha_tensor dk, fmha_tensor dv, int B, int H, int Sq,
                        int Sk, int D, float scale, int mask, int causal_type, void *workspace,
                        size_t workspace_bytes, cudaStream_t stream) {
    if (B < 0 || H <= 0 || Sq < 0 || Sk < 0 || (D != 64 && D != 128)) return FMHA_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !(scale < INFINITY)) return FMHA_ERR_INVALID_ARG;
    if (mask < FMHA_MASK_NONE || mask > FMHA_MASK_CAUSAL) return FMHA_ERR_INVALID_ARG;
    if (causal_type != FMHA_CAUSAL_QBEGIN && causal_type != FMHA_CAUSAL_QEND) return FMHA_ERR_INVALID_ARG;
    if (B == 0 || (Sq == 0 && Sk == 0)) return FMHA_OK;
    if (Sq == 0 || Sk == 0) {
        // no query or no key: every gradient is zero (the side that exists is cleared)
        const size_t n = (size_t)B * (Sq == 0 ? Sk : Sq) * H * D * 2;
        if (Sq == 0) {
            if (!dk.data || !dv.data) return FMHA_ERR_INVALID_ARG;
            if (cudaMemsetAsync(dk.data, 0, n, stream) != cudaSuccess ||
                cudaMemsetAsync(dv.data, 0, n, stream) != cudaSuccess)
                return FMHA_ERR_CUDA;
        } else {
            if (!dq.data) return FMHA_ERR_INVALID_ARG;
            if (cudaMemsetAsync(dq.data, 0, n, stream) != cudaSuccess) return FMHA_ERR_CUDA;
        }
        return FMHA_OK;
    }
    const void *ptrs[9] = {q.data, k.data, v.data, o.data, dout.data, lse, dq.data, dk.data, dv.data};
    const bool need_q = Sq > 0, need_k = Sk > 0;
    const bool need[9] = {need_q, need_k, need_k, need_q, need_q, need_q, need_q, need_k, need_k};
    for (int i = 0; i < 9; ++i)
        if (need[i] && !ptrs[i]) return FMHA_ERR_INVALID_ARG;
    const int dt = q.dtype;
    if (dt != FMHA_F16 && dt != FMHA_BF16 && dt != FMHA_E4M3) return FMHA_ERR_UNSUPPORTED;
    const bool fp8 = dt == FMHA_E4M3;
    const int gdt = fp8 ? FMHA_BF16 : dt;                     // gradients: bf16 for e4m3 inputs
    const fmha_tensor ins[5] = {q, k, v, o, dout}, grads[3] = {dq, dk, dv};
    for (const fmha_tensor &t : ins)
        if (t.data && t.dtype != dt) return FMHA_ERR_UNSUPPORTED;
    for (const fmha_tensor &t : grads)
        if (t.data && t.dtype != gdt) return FMHA_ERR_UNSUPPORTED;
    for (int i = 0; i < 9; ++i) {
        const uintptr_t a = reinterpret_cast<uintptr_t>(ptrs[i]);
        if (i == 5 ? (a & 3u) != 0 : (a & 15u) != 0) return i == 5 ? FMHA_ERR_INVALID_ARG : FMHA_ERR_UNSUPPORTED;
    }
    const size_t need_ws = fmha_bwd_workspace_size_ex(B, H, Sq, Sk, D, dt);
    if (Sq > 0 && (!workspace || workspace_bytes < need_ws || (reinterpret_cast<uintptr_t>(workspace) & 255u)))
        return FMHA_ERR_INVALID_ARG;
    const void *qx = q.data, *kx = k.data, *vx = v.data, *ox = o.data, *dox = dout.data;
    if (fp8) {
        const WidenLayout l = widen_layout(B, H, Sq, Sk, D);
        uint8_t *ws = static_cast<uint8_t *>(workspace);
        Widen w{};
        const void *src[5] = {q.data, o.data, dout.data, k.data, v.data};
        const size_t off[5] = {l.q, l.o, l.dout, l.k, l.v};
        const int64_t rows[5] = {(int64_t)B * Sq, (int64_t)B * Sq, (int64_t)B * Sq, (int64_t)B * Sk,
                                 (int64_t)B * Sk};
        int64_t most = 0;
        for (int t = 0; t < 5; ++t) {
            w.src[t] = static_cast<const uint8_t *>(src[t]);
            w.dst[t] = reinterpret_cast<__nv_bfloat16 *>(ws + off[t]);
            w.n16[t] = rows[t] * H * D / 16;
            most = w.n16[t] > most ? w.n16[t] : most;
        }
        const int64_t blocks = (most + 255) / 256;
        widen_e4m3_kernel<<<(unsigned)(blocks < 4096 ? blocks : 4096), 256, 0, stream>>>(w);
        if (cudaGetLastError() != cudaSuccess) return FMHA_ERR_CUDA;
        qx = w.dst[0];
        ox = w.dst[1];
        dox = w.dst[2];
        kx = w.dst[3];
        vx = w.dst[4];
    }

    BwdParams p{};
    p.q = qx;
    p.k = kx;
    p.v = vx;
    p.o = ox;
    p.dout = dox;
    p.lse = lse;
    p.sq_pad = (Sq + kT - 1) / kT * kT;
    p.nl = static_cast<float *>(workspace);
    p.nd = p.nl + (size_t)B * H * p.sq_pad;
    p.dq = dq.data;
    p.dk = dk.data;
    p.dv = dv.data;
    p.B = B;
    p.H = H;
    p.Sq = Sq;
    p.Sk = Sk;
    p.scale = scale;
    p.c2 = scale * kLog2e;
    p.mask = mask;
    p.causal_type = causal_type;
    p.off = (mask == FMHA_MASK_CAUSAL && causal_type == FMHA_CAUSAL_QEND) ? Sk - Sq : 0;
    const bool bf = gdt == FMHA_BF16;
    return D == 64 ? bwd_launch<64>(p, bf, stream) : bwd_launch<128>(p, bf, stream);
}
