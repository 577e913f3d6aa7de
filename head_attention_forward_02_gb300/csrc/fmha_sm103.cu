// fmha_sm103.cu -- fused attention forward on the sm_103a tensor cores.
//
// O = softmax(scale * Q K^T + mask) V with an online softmax; S and P live in
// tensor memory (TMEM) and never reach HBM.
//
// Design (prior art: "FMHA for Blackwell: Forward" -- two Q tiles per CTA
// ping-ponged between the GEMMs and the softmax, 256 x 128 blocking, fp32
// accumulators; "fmha sm120 : 超越 torch.sdpa(flash-attention-2)" -- TMA
// tiles in swizzled shared memory, a separate barrier for V so its load
// overlaps Q K^T, exp2 with the scale folded into one FMA, lazy rescaling
// of O at a 2^8 threshold, masking only on boundary tiles):
//
//  * persistent CTAs, one per SM; a work unit is (batch, query head, 256
//    query rows) = two 128-row Q tiles; units are taken heaviest first;
//  * warp 8 (one lane) loads Q tiles and a ring of K/V tiles by TMA;
//  * warps 9 and 10 issue the tcgen05.mma of Q tile 0 / 1 (each runs its
//    loop as a whole warp and issues through one elected lane): S_t = Q_t K^T
//    into TMEM (fp32), then O_t += P_t V with P_t read from TMEM (aliasing
//    S_t) and V from shared memory (MN-major); warp 9 owns the TMEM
//    allocation, and the two warps take turns so the pipe sees the order below;
//  * warps 0-3 / 4-7 run the softmax of Q tile 0 / 1, one thread per query
//    row (TMEM lane), and the epilogue of their tile;
//  * the MMA order S0_j, S1_j, PV0_j, S0_{j+1}, PV1_j, S1_{j+1}, ... gives
//    each softmax warpgroup the time of two GEMMs to produce P, and makes
//    "S_t_j complete" imply "PV_t_{j-1} complete", so the softmax warps may
//    rescale O_t in TMEM before publishing P_t_j without another barrier.
//    (Two issuers without the turns were measured slower: the tensor pipe
//    then interleaves the tiles and S_t completes later.)
//
// Every wait is bounded: after g_wait_ns (4 s unless a test sets another
// limit through fmha_set_wait_limit_ns) the waiting thread records
// FMHA_ERR_TIMEOUT in g_status, raises a CTA-wide abort flag, and all roles
// stop issuing work, drain what they issued (bounded), free TMEM and return.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <math.h>
#include <mutex>

#include "fmha_common.h"

namespace fmha {

__device__ int g_status;   // FMHA_OK, or FMHA_ERR_TIMEOUT after a bounded wait expired
// the bounded waits' limit (ns); set from the host through fmha_set_wait_limit_ns
__device__ unsigned long long g_wait_ns = 4000000000ull;
// test hook (fmha_set_test_gate): when set, the producer first waits for a
// flag that nothing sets, so that bounded wait expires and the launch takes
// its failure path
__device__ int g_test_gate;
__device__ int g_test_flag;   // never written

namespace {

constexpr int kTile = 128;                 // query rows per Q tile, keys per K/V tile
constexpr int kUnitRows = 2 * kTile;       // query rows per work unit
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;                // issues Q tile 0's MMAs; owns the TMEM allocation
constexpr int kMmaWarp1 = 10;              // issues Q tile 1's MMAs
static_assert(kMmaWarp1 == kMmaWarp + 1, "issuing warp t is kMmaWarp + t");
constexpr int kThreads = 352;              // softmax warps 0-7, producer warp 8, MMA warps 9-10
constexpr uint32_t kTmemCols = 512;
constexpr unsigned long long kTimeoutNs = 4000000000ull;
constexpr unsigned long long kDrainNs = 200000000ull;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.0f;       // rescale O when the max grows by > 2^8

enum Elem { kF16 = 0, kBF16 = 1, kE4M3 = 2 };

template <int D_, int ELEM_>
struct Cfg {
    static constexpr int D = D_;
    static constexpr int ELEM = ELEM_;
    static constexpr bool FP8 = ELEM == kE4M3;
    static constexpr int E = FP8 ? 1 : 2;                 // bytes per element
    static constexpr int ROW_BYTES = D * E;
    static constexpr int SW = ROW_BYTES >= 128 ? 128 : ROW_BYTES;   // swizzle span (bytes)
    static constexpr int PANELS = ROW_BYTES / SW;         // 128-byte column panels per row
    static constexpr int BOX_D = SW / E;                  // elements per panel row
    static constexpr int PANEL_BYTES = kTile * SW;
    static constexpr int TILE_BYTES = kTile * ROW_BYTES;
    static constexpr uint64_t SW_CODE = SW == 128 ? 2 : (SW == 64 ? 4 : 6);
    static constexpr int SBO = 8 * SW;                    // one 8-row swizzle atom
    static constexpr int MMA_K = FP8 ? 32 : 16;           // K of one tcgen05.mma
    static constexpr int KSTEP_BYTES = MMA_K * E;         // 32 bytes
    static constexpr int QK_STEPS = D / MMA_K;
    static constexpr int PV_STEPS = kTile / MMA_K;
    static constexpr int NS = TILE_BYTES <= 8192 ? 8 : (TILE_BYTES <= 16384 ? 6 : 4);
    // Head dims up to 64 leave TMEM for a P buffer per Q tile, apart from its
    // S columns (PSEP): S_t,j+1 may then overwrite S_t as soon as the softmax
    // warps hold S_t,j in registers, instead of after PV_t,j has read P_t,j
    // from those columns, so the next S is computed while the softmax works.
    // At D = 128 the two O accumulators take the room and P aliases S.
    static constexpr bool PSEP = D <= 64;
    // 16-bit inputs pair the ring: stage i holds V_{j-1} and K_j behind one
    // barrier, so an issuing warp waits and releases once per key step
    // (measured +2% at D=128); e4m3 keeps one tile per stage, where V_j is
    // not held back by K_{j+1} (pairing measured -3% there).  With separate
    // P buffers an issuing warp takes K_{j+1} before V_j, the order of a
    // paired stage, so those pair the ring for every input type.
    static constexpr bool PAIRED = !FP8 || PSEP;
    static constexpr int NSTAGE = PAIRED ? NS / 2 : NS;   // ring stages (barrier pairs)
    // An issuing warp hands the turn to the other one this many MMAs before
    // the end of an S group, hiding the other warp's wake-up behind
    // MMAs still to issue (16-bit: +6% at D=128).  The e4m3 key step is
    // softmax-bound, and there letting the other tile's MMAs in ahead of the
    // last S MMAs costs more than the hand-off (measured -2% to -5%).
    static constexpr int TURN_EARLY = FP8 ? 0 : 2;
    static constexpr int TURN_AT = QK_STEPS - 1 - TURN_EARLY > 0 ? QK_STEPS - 1 - TURN_EARLY : 0;
    static constexpr int S_COL0 = 0, S_COL1 = kTile;
    static constexpr int O_COL0 = 2 * kTile, O_COL1 = 2 * kTile + D;
    static constexpr int P_COL0 = PSEP ? O_COL1 + D : S_COL0, P_COL1 = PSEP ? P_COL0 + 64 : S_COL1;
    static_assert(!PSEP || P_COL1 + 64 <= (int)kTmemCols, "TMEM budget of the P buffers");
    static constexpr int BAR_BYTES = 512;
    // O staging for the TMA store of the epilogue: per softmax warp 32 rows x
    // one swizzle panel (a row of several panels goes out panel by panel)
    static constexpr int STG_WARP = 32 * SW;
    static constexpr int STG_BYTES = 8 * STG_WARP;
    static constexpr int SMEM_USED = 2 * TILE_BYTES + NS * TILE_BYTES + STG_BYTES + BAR_BYTES;
    // at least 120 KB so that a second CTA can never share the SM (TMEM is
    // allocated whole), plus 1 KB to align the tiles for the 128-byte swizzle
    static constexpr int SMEM_BYTES = (SMEM_USED < 120 * 1024 ? 120 * 1024 : SMEM_USED) + 1024;
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
    static_assert(O_COL1 + D <= (int)kTmemCols, "TMEM budget");
    // instruction descriptor fields (kind::f16: 0 = f16, 1 = bf16; kind::f8f6f4: 0 = e4m3)
    static constexpr uint32_t AB_FMT = ELEM == kBF16 ? 1u : 0u;
    static constexpr uint32_t idesc(int n, bool b_mn_major) {
        return (1u << 4)                        // D: f32
               | (AB_FMT << 7) | (AB_FMT << 10)  // A, B formats
               | ((b_mn_major ? 1u : 0u) << 16)  // B major-ness
               | ((uint32_t)(n >> 3) << 17)      // N >> 3
               | ((uint32_t)(kTile >> 4) << 24); // M >> 4
    }
};

struct Bars {
    uint64_t q_full[2], q_empty[2], s_full[2], p_half[2], p_full[2], o_full[2], drain;
    uint64_t turn[2];          // issue turn of the issuing warp of Q tile t
    uint64_t s_free[2];        // separate P buffers: the softmax warps hold S_t in registers
    uint64_t pv_done[2];       // separate P buffers: PV_t complete (P_t and O_t free)
    uint64_t kv_full[8], kv_empty[8];
    uint32_t tmem_base;
    int abort;
};

// ---------------------------------------------------------------------------
// PTX wrappers (mbarrier, TMA, tcgen05)
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
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n"
        "}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Slow path of a bounded wait: poll until the phase completes, the CTA aborts,
// or g_wait_ns pass (then record the timeout and raise the abort flag).
__device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, volatile int *abort_flag) {
    const unsigned long long t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63) == 0) {
            if (*abort_flag) return false;
            if (globaltimer() - t0 > g_wait_ns) {
                *abort_flag = 1;
                atomicExch(&g_status, FMHA_ERR_TIMEOUT);
                return false;
            }
        }
    }
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    return mbar_wait_slow(bar, parity, abort_flag);
}

// Bounded wait that ignores the abort flag (used only while draining).
__device__ __noinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity) {
    const unsigned long long t0 = globaltimer();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer() - t0 > kDrainNs) return false;
    }
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int c0, int c1, int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
        : "memory");
}

// O is written once and read by nobody in this kernel: its lines are marked
// first to leave L2, ahead of the K/V tiles other units still read
__device__ __forceinline__ uint64_t evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, uint32_t src, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group.L2::cache_hint [%0, {%2, %3, %4}], [%1], %5;" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(c0), "r"(c1), "r"(c2), "l"(evict_first_policy())
                 : "memory");
}

__device__ __forceinline__ void tma_store_4d(const CUtensorMap *map, uint32_t src, int c0, int c1, int c2, int c3) {
    asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.bulk_group.L2::cache_hint [%0, {%2, %3, %4, %5}], [%1], %6;" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "l"(evict_first_policy())
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// this thread's bulk stores have read their shared-memory source
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// this thread's bulk stores are complete
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// loads with an L2 policy (Q: read by one unit only)
__device__ __forceinline__ void tma_load_3d_hint(uint32_t dst, const CUtensorMap *map, uint32_t bar, int c0, int c1,
                                                 int c2, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar), "l"(pol)
        : "memory");
}

__device__ __forceinline__ void tma_load_4d_hint(uint32_t dst, const CUtensorMap *map, uint32_t bar, int c0, int c1,
                                                 int c2, int c3, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar), "l"(pol)
        : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor (start address, leading / stride byte
// offsets in 16-byte units, descriptor version 1, swizzle mode) as two 32-bit
// words.  The low word holds the start address (14 bits) and the leading
// byte offset; adding (bytes >> 4) to it moves the start address without
// touching anything else as long as the address stays in the 256 KB window,
// which shared memory does.
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
template <bool FP8>
__device__ __forceinline__ void mma_ss_e(uint32_t d, uint32_t a_lo, uint32_t b_lo, uint32_t hi, uint32_t idesc,
                                         uint32_t acc) {
    if constexpr (FP8) {
        asm volatile(
            "{\n.reg .pred p, e;\n.reg .b64 da, db;\nsetp.ne.b32 p, %4, 0;\nelect.sync _|e, 0xffffffff;\n"
            "mov.b64 da, {%1, %3};\nmov.b64 db, {%2, %3};\n"
            "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], da, db, %5, p;\n}\n" ::"r"(d),
            "r"(a_lo), "r"(b_lo), "r"(hi), "r"(acc), "r"(idesc)
            : "memory");
    } else {
        asm volatile(
            "{\n.reg .pred p, e;\n.reg .b64 da, db;\nsetp.ne.b32 p, %4, 0;\nelect.sync _|e, 0xffffffff;\n"
            "mov.b64 da, {%1, %3};\nmov.b64 db, {%2, %3};\n"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, p;\n}\n" ::"r"(d),
            "r"(a_lo), "r"(b_lo), "r"(hi), "r"(acc), "r"(idesc)
            : "memory");
    }
}

template <bool FP8>
__device__ __forceinline__ void mma_ts_e(uint32_t d, uint32_t a, uint32_t b_lo, uint32_t hi, uint32_t idesc,
                                         uint32_t acc) {
    if constexpr (FP8) {
        asm volatile(
            "{\n.reg .pred p, e;\n.reg .b64 db;\nsetp.ne.b32 p, %4, 0;\nelect.sync _|e, 0xffffffff;\n"
            "mov.b64 db, {%2, %3};\n"
            "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], db, %5, p;\n}\n" ::"r"(d),
            "r"(a), "r"(b_lo), "r"(hi), "r"(acc), "r"(idesc)
            : "memory");
    } else {
        asm volatile(
            "{\n.reg .pred p, e;\n.reg .b64 db;\nsetp.ne.b32 p, %4, 0;\nelect.sync _|e, 0xffffffff;\n"
            "mov.b64 db, {%2, %3};\n"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], db, %5, p;\n}\n" ::"r"(d),
            "r"(a), "r"(b_lo), "r"(hi), "r"(acc), "r"(idesc)
            : "memory");
    }
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

// Bounded wait by a whole warp: true in every lane, or false in every lane.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag) {
    const bool r = mbar_wait(bar, parity, abort_flag);
    return __all_sync(0xffffffffu, r);
}

// The same bounded wait with its polling loop inlined: for call sites where
// many values are live (a call to the out-of-line slow path would make the
// compiler save them all around it).
__device__ __forceinline__ bool warp_wait_inline(uint32_t bar, uint32_t parity, volatile int *abort_flag) {
    bool r = mbar_try_wait(bar, parity);
    if (!r) {
        const unsigned long long t0 = globaltimer();
        for (uint32_t it = 1;; ++it) {
            if ((r = mbar_try_wait(bar, parity))) break;
            if ((it & 63) == 0) {
                if (*abort_flag) break;
                if (globaltimer() - t0 > g_wait_ns) {
                    *abort_flag = 1;
                    atomicExch(&g_status, FMHA_ERR_TIMEOUT);
                    break;
                }
            }
        }
    }
    return __all_sync(0xffffffffu, r);
}



__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Packed pairs of fp32 (one 64-bit register pair) for the f32x2 FMA / add.
__device__ __forceinline__ uint64_t pack_f2(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}

__device__ __forceinline__ void unpack_f2(uint64_t v, float &a, float &b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}

__device__ __forceinline__ uint64_t fma_f2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.ftz.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__device__ __forceinline__ uint64_t add_f2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.ftz.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Load 32 consecutive TMEM columns of this thread's lane (32x32b shape).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr));
}

// Wait for this thread's outstanding TMEM loads; the register operands tie the
// loaded values to the wait so no use of them can be scheduled before it.
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}

// The same wait, also taking a value computed before it as an operand, so that
// the computation stays ahead of the wait and overlaps the loads in flight.
__device__ __forceinline__ void tmem_wait_ld_after(uint32_t (&r)[32], float &v) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31]), "+f"(v)
                 :
                 : "memory");
}



// Store 16 consecutive TMEM columns of this thread's lane (32x32b shape).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};"
                 :
                 : "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
                   "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
                 : "memory");
}

// Store 32 consecutive TMEM columns of this thread's lane (32x32b shape).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};"
                 :
                 : "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
                 : "memory");
}

// ---------------------------------------------------------------------------
// Element packing
// ---------------------------------------------------------------------------

template <int ELEM>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    if constexpr (ELEM == kBF16) {
        __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&v);
    } else {
        __half2 v = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&v);
    }
}

// four values to e4m3 (round to nearest even, saturating), first value in the low byte
__device__ __forceinline__ uint32_t pack4_e4m3(float a, float b, float c, float d) {
    const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
    return lo | (hi << 16);
}

// ---------------------------------------------------------------------------
// Work units: (batch, query head, 256 query rows), heaviest first for causal
// ---------------------------------------------------------------------------

struct Unit {
    int b, h, g, q0;      // batch, query head, kv head, first query row of the unit
    int sq, sk;           // sequence lengths
    int q_row, k_row;     // row of the sequence's first token in the stored tensors
    int n[2], nu[2];      // per Q tile: end of its key tiles in this work item / unmasked ones
    int j0, j1;           // key tiles [j0, j1) of this work item (split-KV: one range of several)
    int split;            // split index (0 without split-KV)
};

// Query head and first row of Q tile t of a unit: rows q0 + 128 t of head h,
// or, with head pairs, head h + t over rows [q0, q0 + 128)
template <bool HP>
__device__ __forceinline__ int tile_head(const Unit &U, int t) { return HP ? U.h + t : U.h; }
template <bool HP>
__device__ __forceinline__ int tile_row0(const Unit &U, int t) { return HP ? U.q0 : U.q0 + t * kTile; }

// Unit taken by this CTA in round r: CTAs sweep the (heaviest-first) unit
// list in alternating directions, which balances causal work to within a
// fraction of a unit without a shared work counter.
__device__ __forceinline__ int unit_of_round(int r) {
    return r * gridDim.x + ((r & 1) ? gridDim.x - 1 - blockIdx.x : blockIdx.x);
}

struct Cursor {                  // varlen decoding state (units are decoded in increasing order)
    int b = 0, base = 0;         // sequence-major order: current sequence, index of its first unit
    bool init = false;           // block-level order (causal):
    int q = 0, qbase = 0, qcnt = 0;  // current 256-row block index, its first unit, sequences that have it
};

// 256-row query blocks of packed sequence b
__device__ __forceinline__ int seq_blocks(const Params &p, int b) {
    return (p.cu_q[b + 1] - p.cu_q[b] + kUnitRows - 1) / kUnitRows;
}

__device__ __forceinline__ int seqs_with_block(const Params &p, int q) {
    int n = 0;
    for (int b = 0; b < p.B; ++b) n += seq_blocks(p, b) > q;
    return n;
}

template <bool HP>
__device__ __forceinline__ bool decode_unit(const Params &p, int u, Cursor &cur, Unit &U) {
    int b, h, qb;
    if constexpr (HP) {
        // head pairs (fixed length, Sq <= 128, even query group): one unit
        // per (batch, query heads 2i and 2i + 1); both Q tiles cover rows
        // [0, Sq) and read the same kv head's K/V
        if (u >= p.B * (p.H / 2)) return false;
        b = u / (p.H / 2);
        h = 2 * (u - b * (p.H / 2));
        U.b = b;
        U.h = h;
        U.g = h / p.group;
        U.q0 = 0;
        U.sq = p.Sq;
        U.sk = p.Sk;
        U.q_row = b * p.Sq;
        U.k_row = b * p.Sk;
        kv_tile_range(0, kTile, U.sq, U.sk, p.mask, p.causal_type, kTile, &U.n[0], &U.nu[0]);
        U.n[1] = U.n[0];
        U.nu[1] = U.nu[0];
        return true;
    }
    if (!p.varlen) {
        const int nqb = (p.Sq + kUnitRows - 1) / kUnitRows;
        const int per = p.B * p.H;
        if (u >= per * nqb) return false;
        if (p.mask == FMHA_MASK_CAUSAL) {
            // causal work grows with the block index: block level by block
            // level, deepest first, across all heads (heaviest first)
            const int r = u / per, rem = u - r * per;
            b = rem / p.H;
            h = rem - b * p.H;
            qb = nqb - 1 - r;
        } else {
            // every unit has the same work: all blocks of one head in a row,
            // so the CTAs in flight share that head's K/V in L2
            const int bh = u / nqb;
            qb = u - bh * nqb;
            b = bh / p.H;
            h = bh - b * p.H;
        }
        U.sq = p.Sq;
        U.sk = p.Sk;
        U.q_row = b * p.Sq;
        U.k_row = b * p.Sk;
    } else if (p.mask == FMHA_MASK_CAUSAL) {
        // Causal work grows with the block index, so units go block level by
        // block level, deepest first, across all sequences (heaviest first).
        if (!cur.init) {
            int mx = 0;
            for (int bb = 0; bb < p.B; ++bb) mx = imax(mx, seq_blocks(p, bb));
            cur.init = true;
            cur.q = mx - 1;
            cur.qbase = 0;
            cur.qcnt = cur.q >= 0 ? seqs_with_block(p, cur.q) : 0;
        }
        while (cur.q >= 0 && u >= cur.qbase + cur.qcnt * p.H) {
            cur.qbase += cur.qcnt * p.H;
            --cur.q;
            cur.qcnt = cur.q >= 0 ? seqs_with_block(p, cur.q) : 0;
        }
        if (cur.q < 0) return false;
        const int rem = u - cur.qbase;
        int k = rem / p.H;
        h = rem - k * p.H;
        b = 0;
        for (int bb = 0; bb < p.B; ++bb) {
            if (seq_blocks(p, bb) > cur.q) {
                if (k == 0) { b = bb; break; }
                --k;
            }
        }
        qb = cur.q;
        U.q_row = p.cu_q[b];
        U.sq = p.cu_q[b + 1] - U.q_row;
        U.k_row = p.cu_k[b];
        U.sk = p.cu_k[b + 1] - U.k_row;
    } else {
        int bb = cur.b, base = cur.base;
        for (;;) {
            if (bb >= p.B) {
                cur.b = bb;
                cur.base = base;
                return false;
            }
            const int cnt = seq_blocks(p, bb) * p.H;
            if (u < base + cnt) break;
            base += cnt;
            ++bb;
        }
        cur.b = bb;
        cur.base = base;
        b = bb;
        const int rem = u - base;
        U.q_row = p.cu_q[b];
        U.sq = p.cu_q[b + 1] - U.q_row;
        U.k_row = p.cu_k[b];
        U.sk = p.cu_k[b + 1] - U.k_row;
        const int nqb = (U.sq + kUnitRows - 1) / kUnitRows;
        qb = nqb - 1 - rem / p.H;
        h = rem % p.H;
    }
    U.b = b;
    U.h = h;
    U.g = h / p.group;
    U.q0 = qb * kUnitRows;
    kv_tile_range(U.q0, kTile, U.sq, U.sk, p.mask, p.causal_type, kTile, &U.n[0], &U.nu[0]);
    kv_tile_range(U.q0 + kTile, kTile, U.sq, U.sk, p.mask, p.causal_type, kTile, &U.n[1], &U.nu[1]);
    return true;
}

// Work item u = unit u / num_splits, key range number u % num_splits: the
// unit's key tiles [0, max(n0, n1)) are cut into num_splits near-equal
// contiguous ranges; tile t then covers [j0, min(n_t, j1)) and is active
// when that range is not empty.  Without split-KV, j0 = 0 and j1 = max(n0, n1).
// The same decoder as an out-of-line call: the e4m3 D=128 kernels keep fewer
// values live through their softmax loops that way (measured +1.2% to +2.5%;
// at D=64 it measured -1.6%, and the 16-bit kernels do not gain)
template <bool HP>
__device__ __noinline__ bool decode_unit_call(const Params &p, int u, Cursor &cur, Unit &U) {
    return decode_unit<HP>(p, u, cur, U);
}

template <bool SPLIT, bool HP, bool OUTLINE = false>
__device__ __forceinline__ bool decode_work(const Params &p, int u, Cursor &cur, Unit &U) {
    const int ns = SPLIT ? p.num_splits : 1;      // a constant 1 folds the split arithmetic away
    if (OUTLINE ? !decode_unit_call<HP>(p, u / ns, cur, U) : !decode_unit<HP>(p, u / ns, cur, U)) return false;
    const int nmax = imax(U.n[0], U.n[1]);
    U.split = u % ns;
    U.j0 = (int)((int64_t)nmax * U.split / ns);
    U.j1 = (int)((int64_t)nmax * (U.split + 1) / ns);
    U.n[0] = imin(U.n[0], U.j1);
    U.n[1] = imin(U.n[1], U.j1);
    return true;
}

// ---------------------------------------------------------------------------
// Producer: Q tiles and the K/V ring, by TMA (one lane)
// ---------------------------------------------------------------------------

template <class C, bool SPLIT, bool HP>
__device__ void producer(const Params &p, const CUtensorMap *tmQ, const CUtensorMap *tmK,
                         const CUtensorMap *tmV, uint8_t *sQ, uint8_t *sKV, Bars *bars) {
    volatile int *abort_flag = &bars->abort;
    prefetch_tmap(tmQ);
    prefetch_tmap(tmK);
    prefetch_tmap(tmV);
    uint32_t fill = 0, qload[2] = {0, 0};
    bool ok = true;
    if (g_test_gate) {
        // a flag nothing sets: the wait runs out, records the timeout and
        // raises the abort flag; no copy has been issued yet
        const volatile int *flag = &g_test_flag;
        const unsigned long long t0 = globaltimer();
        for (uint32_t it = 1; !*flag; ++it) {
            if ((it & 63) == 0 && (*abort_flag || globaltimer() - t0 > g_wait_ns)) {
                *abort_flag = 1;
                atomicExch(&g_status, FMHA_ERR_TIMEOUT);
                break;
            }
        }
        ok = false;
    }
    Cursor cur;
    for (int r = 0; ok; ++r) {
        Unit U;
        if (!decode_work<SPLIT, HP, C::FP8 && C::D == 128>(p, unit_of_round(r), cur, U)) break;
        for (int t = 0; t < 2; ++t) {
            if (U.n[t] <= U.j0) continue;                 // tile inactive in this work item
            if (qload[t] > 0 &&
                !mbar_wait(smem_u32(&bars->q_empty[t]), (qload[t] - 1) & 1, abort_flag)) {
                ok = false;
                break;
            }
            const uint32_t fb = smem_u32(&bars->q_full[t]);
            mbar_expect_tx(fb, C::TILE_BYTES);
            const uint32_t dst = smem_u32(sQ + t * C::TILE_BYTES);
            const int row = tile_row0<HP>(U, t), qh = tile_head<HP>(U, t);
            // a Q tile is read by this unit only: first to leave L2, ahead of K/V
            const uint64_t pol = evict_first_policy();
#pragma unroll
            for (int pn = 0; pn < C::PANELS; ++pn) {
                if (p.varlen)
                    tma_load_3d_hint(dst + pn * C::PANEL_BYTES, tmQ, fb, pn * C::BOX_D, qh, U.q_row + row, pol);
                else
                    tma_load_4d_hint(dst + pn * C::PANEL_BYTES, tmQ, fb, pn * C::BOX_D, qh, row, U.b, pol);
            }
            ++qload[t];
        }
        if constexpr (C::PAIRED) {
            // fill i of a work item holds V_{j0+i-1} (none for i = 0) and
            // K_{j0+i} (none for the last fill)
            for (int i = 0; i <= U.j1 - U.j0 && U.j0 < U.j1 && ok; ++i) {
                const int st = fill % C::NSTAGE;
                const uint32_t rnd = fill / C::NSTAGE;
                if (rnd > 0 && !mbar_wait(smem_u32(&bars->kv_empty[st]), (rnd - 1) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                const int jk = U.j0 + i, jv = U.j0 + i - 1;
                const bool has_k = jk < U.j1, has_v = i > 0;
                const uint32_t fb = smem_u32(&bars->kv_full[st]);
                mbar_expect_tx(fb, (has_k + has_v) * C::TILE_BYTES);
                const uint32_t dst = smem_u32(sKV + st * 2 * C::TILE_BYTES);
#pragma unroll
                for (int kv = 0; kv < 2; ++kv) {
                    if (kv ? !has_v : !has_k) continue;
                    const CUtensorMap *m = kv ? tmV : tmK;
                    const int j = kv ? jv : jk;
                    const uint32_t d = dst + kv * C::TILE_BYTES;
#pragma unroll
                    for (int pn = 0; pn < C::PANELS; ++pn) {
                        if (p.varlen)
                            tma_load_3d(d + pn * C::PANEL_BYTES, m, fb, pn * C::BOX_D, U.g, U.k_row + j * kTile);
                        else
                            tma_load_4d(d + pn * C::PANEL_BYTES, m, fb, pn * C::BOX_D, U.g, j * kTile, U.b);
                    }
                }
                ++fill;
            }
        } else {
            for (int j = U.j0; j < U.j1 && ok; ++j) {
                for (int kv = 0; kv < 2; ++kv) {
                    const int st = fill % C::NSTAGE;
                    const uint32_t rnd = fill / C::NSTAGE;
                    if (rnd > 0 && !mbar_wait(smem_u32(&bars->kv_empty[st]), (rnd - 1) & 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = smem_u32(&bars->kv_full[st]);
                    mbar_expect_tx(fb, C::TILE_BYTES);
                    const uint32_t dst = smem_u32(sKV + st * C::TILE_BYTES);
                    const CUtensorMap *m = kv ? tmV : tmK;
#pragma unroll
                    for (int pn = 0; pn < C::PANELS; ++pn) {
                        if (p.varlen)
                            tma_load_3d(dst + pn * C::PANEL_BYTES, m, fb, pn * C::BOX_D, U.g,
                                        U.k_row + j * kTile);
                        else
                            tma_load_4d(dst + pn * C::PANEL_BYTES, m, fb, pn * C::BOX_D, U.g, j * kTile, U.b);
                    }
                    ++fill;
                }
            }
        }
    }
    if (ok) {
        // every stage's last release and every Q tile's last release must have
        // arrived before the CTA may exit
        for (int st = 0; st < C::NSTAGE; ++st) {
            const uint32_t nf = fill > (uint32_t)st ? (fill - st + C::NSTAGE - 1) / C::NSTAGE : 0;
            if (nf && !mbar_wait(smem_u32(&bars->kv_empty[st]), (nf - 1) & 1, abort_flag)) break;
        }
        for (int t = 0; t < 2; ++t)
            if (qload[t] && !mbar_wait(smem_u32(&bars->q_empty[t]), (qload[t] - 1) & 1, abort_flag))
                break;
    } else {
        // aborted: let the copies already issued land before the CTA exits
        const uint32_t first = fill > (uint32_t)C::NSTAGE ? fill - C::NSTAGE : 0;
        for (uint32_t f = first; f < fill; ++f)
            mbar_wait_drain(smem_u32(&bars->kv_full[f % C::NSTAGE]), (f / C::NSTAGE) & 1);
        for (int t = 0; t < 2; ++t)
            if (qload[t]) mbar_wait_drain(smem_u32(&bars->q_full[t]), (qload[t] - 1) & 1);
    }
}

// ---------------------------------------------------------------------------
// MMA issuers (warps 9 and 10, one elected lane each)
// ---------------------------------------------------------------------------

template <class C, bool SPLIT, bool HP>
__device__ void mma_issuer(const Params &p, uint8_t *sQ, uint8_t *sKV, Bars *bars, uint32_t tmem_any, int t) {
    // Two warps issue the MMAs, warp t for Q tile t, and take turns so that
    // the tensor pipe sees the order S0_j0, S1_j0, then per key step
    // PV0_j S0_j+1, PV1_j S1_j+1: each S_t lands right behind its PV_t and the
    // other tile's work fills the pipe while tile t's softmax runs.  A
    // tcgen05.mma holds its issuing thread for most of its 64 pipe cycles, so
    // one issuer alone cannot also do the commits and barrier waits between
    // groups without starving the shallow tensor queue; with two issuers
    // that bookkeeping runs while the other one issues.
    // The whole warp runs this loop, converged and with warp-uniform values;
    // one elected lane issues each MMA, commit and arrive, so the operand
    // words stay in uniform registers.
    volatile int *abort_flag = &bars->abort;
    const uint32_t tmem = __shfl_sync(0xffffffffu, tmem_any, 0);   // the same in every lane
    constexpr uint32_t kIdS = C::idesc(kTile, false);
    constexpr uint32_t kIdPV = C::idesc(C::D, true);
    uint32_t cons = 0, qc = 0, pc = 0, hc = 0, tc = 0;
    bool ok = true;
    Cursor cur;

    // Descriptor words are computed once; each MMA then only adds a
    // compile-time byte offset to the low word.
    constexpr uint32_t kHi = desc_hi(C::SBO, (uint32_t)C::SW_CODE);
    constexpr uint32_t kTileStep = C::TILE_BYTES >> 4;
    const uint32_t q_lo = desc_lo(smem_u32(sQ), 16) + t * kTileStep;  // K-major: LBO unused
    const uint32_t k_lo = desc_lo(smem_u32(sKV), 16);
    const uint32_t v_lo = desc_lo(smem_u32(sKV), C::PANEL_BYTES);    // MN-major: LBO = panel stride
    const uint32_t s_tm = tmem + (t ? C::S_COL1 : C::S_COL0);
    const uint32_t o_tm = tmem + (t ? C::O_COL1 : C::O_COL0);
    const uint32_t s_full = smem_u32(&bars->s_full[t]), q_empty = smem_u32(&bars->q_empty[t]);
    const uint32_t o_full = smem_u32(&bars->o_full[t]);
    const uint32_t p_half = smem_u32(&bars->p_half[t]), p_full = smem_u32(&bars->p_full[t]);
    const uint32_t my_turn = smem_u32(&bars->turn[t]), next_turn = smem_u32(&bars->turn[t ^ 1]);

    auto pass_turn = [&]() { mbar_arrive_e(next_turn); };
    // S_t = Q_t K^T: both operands K-major; each k-step advances 32 bytes
    // within a 128-byte swizzled panel row, then moves to the next panel.
    // The issue turn passes to the other lane within this group (TURN_AT).
    auto issue_s = [&](int st) {
        // K tile: whole stage, or the first half of a paired stage
        const uint32_t b = k_lo + st * (C::PAIRED ? 2 : 1) * kTileStep;
#pragma unroll
        for (int kk = 0; kk < C::QK_STEPS; ++kk) {
            const uint32_t off =
                ((kk * C::KSTEP_BYTES / C::SW) * C::PANEL_BYTES + (kk * C::KSTEP_BYTES) % C::SW) >> 4;
            mma_ss_e<C::FP8>(s_tm, q_lo + off, b + off, kHi, kIdS, kk > 0 ? 1u : 0u);
            if (kk == C::TURN_AT) pass_turn();
        }
    };
    // O_t (+)= P_t V over one half of the keys (hf = 0: keys 0-63, 1: 64-127):
    // P from TMEM (aliasing S_t), V MN-major (keys are the K dimension, head
    // dim the N dimension spread over PANELS panels).
    auto issue_pv_half = [&](int st, int hf, bool acc) {
        // V tile: whole stage, or the second half of a paired stage
        const uint32_t b = v_lo + (C::PAIRED ? st * 2 + 1 : st) * kTileStep;
        constexpr int H = C::PV_STEPS / 2;
#pragma unroll
        for (int k = 0; k < H; ++k) {
            const int kk = hf * H + k;
            mma_ts_e<C::FP8>(o_tm, s_tm + kk * (C::MMA_K * C::E / 4), b + ((kk * C::MMA_K * C::SW) >> 4), kHi,
                             kIdPV, (acc || kk > 0) ? 1u : 0u);
        }
    };
    // TMA writes and tensor-core reads of shared memory are both async-proxy
    // operations ordered by the mbarrier: no tcgen05 fence is needed here.
    // Both lanes consume every ring stage and each releases it once.
    auto next_kv = [&](int &st) -> bool {
        st = cons % C::NSTAGE;
        const bool r = warp_wait(smem_u32(&bars->kv_full[st]), (cons / C::NSTAGE) & 1, abort_flag);
        ++cons;
        return r;
    };
    // P_t was written to TMEM by the softmax threads (tcgen05.st): order this
    // thread's MMAs after their fence::before_thread_sync + arrive.
    auto wait_p = [&](uint32_t bar, uint32_t &cnt) -> bool {
        const bool r = warp_wait(bar, cnt & 1, abort_flag);
        ++cnt;
        if (r) tc_fence_after();
        return r;
    };
    auto take_turn = [&]() -> bool {
        const bool r = warp_wait(my_turn, tc & 1, abort_flag);
        ++tc;
        return r;
    };

    for (int r = 0; ok; ++r) {
        Unit U;
        if (!decode_work<SPLIT, HP, C::FP8 && C::D == 128>(p, unit_of_round(r), cur, U)) break;
        const int n = t ? U.n[1] : U.n[0], j0 = U.j0, jn = U.j1;
        if (j0 >= jn) continue;
        if (n > j0) {
            ok = warp_wait(smem_u32(&bars->q_full[t]), qc & 1, abort_flag);
            ++qc;
        }
        int kst;
        if (!ok || !next_kv(kst) || !take_turn()) { ok = false; break; }
        // the previous unit's epilogue read O_t from TMEM before its softmax
        // warps published this unit's first P_t, so no wait is needed here
        if (n > j0) issue_s(kst);
        else pass_turn();
        if (n > j0) {
            tc_commit_e(s_full);
            if (n == j0 + 1) tc_commit_e(q_empty);
        }
        tc_commit_e(smem_u32(&bars->kv_empty[kst]));
        for (int j = j0; j < jn; ++j) {
            // paired ring: one stage holds V_j and K_{j+1}; otherwise V_j,
            // then K_{j+1} in the next stage (when a next key tile exists)
            int v_st, k_st = 0;
            if (!next_kv(v_st)) { ok = false; break; }
            if constexpr (C::PAIRED) k_st = v_st;
            else if (j + 1 < jn && !next_kv(k_st)) { ok = false; break; }
            const bool act = j < n, more = j + 1 < n;
            // P_t is published in two halves: PV over keys 0-63 starts once
            // the first half is in TMEM, while the softmax computes the
            // second; S_t,j+1 overwrites P_t after both PV halves in pipe order
            if (act && !wait_p(p_half, hc)) { ok = false; break; }
            if (!take_turn()) { ok = false; break; }
            if (act) {
                issue_pv_half(v_st, 0, j > j0);
                if (!wait_p(p_full, pc)) { ok = false; break; }
                issue_pv_half(v_st, 1, true);
                if (more) issue_s(k_st);
            }
            if (!act || !more) pass_turn();
            if (act) {
                if (!more) {
                    tc_commit_e(o_full);
                } else {
                    tc_commit_e(s_full);
                    if (j + 2 == n) tc_commit_e(q_empty);
                }
            }
            tc_commit_e(smem_u32(&bars->kv_empty[v_st]));
            if (!C::PAIRED && j + 1 < jn) tc_commit_e(smem_u32(&bars->kv_empty[k_st]));
        }
    }
    // no tensor-core operation may be in flight when TMEM is released
    tc_commit_e(smem_u32(&bars->drain));
    mbar_wait_drain(smem_u32(&bars->drain), 0);
}

// Issuing warp t with separate P buffers (head dims 32 and 64).  Per key step
// j it issues S_t,j+1 as soon as the softmax warps signal that they hold
// S_t,j in registers (s_free), then PV_t,j from the P buffer once P_t,j is
// published; the paired ring stage j+1 holds both K_j+1 and V_j.  The two
// warps run free: S is issued about a softmax step ahead of its use, so the
// pipe order between the tiles matters little.  PV_t,j completes pv_done[t],
// which the softmax warps wait for before they overwrite P_t or rescale O_t.
template <class C, bool SPLIT, bool HP>
__device__ void mma_issuer_psep(const Params &p, uint8_t *sQ, uint8_t *sKV, Bars *bars, uint32_t tmem_any,
                                int t) {
    volatile int *abort_flag = &bars->abort;
    const uint32_t tmem = __shfl_sync(0xffffffffu, tmem_any, 0);   // the same in every lane
    constexpr uint32_t kIdS = C::idesc(kTile, false);
    constexpr uint32_t kIdPV = C::idesc(C::D, true);
    constexpr uint32_t kHi = desc_hi(C::SBO, (uint32_t)C::SW_CODE);
    constexpr uint32_t kTileStep = C::TILE_BYTES >> 4;
    static_assert(C::PAIRED, "separate P buffers consume the ring in paired order");
    const uint32_t q_lo = desc_lo(smem_u32(sQ), 16) + t * kTileStep;  // K-major: LBO unused
    const uint32_t k_lo = desc_lo(smem_u32(sKV), 16);
    const uint32_t v_lo = desc_lo(smem_u32(sKV), C::PANEL_BYTES);    // MN-major: LBO = panel stride
    const uint32_t s_tm = tmem + (t ? C::S_COL1 : C::S_COL0);
    const uint32_t o_tm = tmem + (t ? C::O_COL1 : C::O_COL0);
    const uint32_t p_tm = tmem + (t ? C::P_COL1 : C::P_COL0);
    const uint32_t s_full = smem_u32(&bars->s_full[t]), q_empty = smem_u32(&bars->q_empty[t]);
    const uint32_t s_free = smem_u32(&bars->s_free[t]), pv_done = smem_u32(&bars->pv_done[t]);
    const uint32_t o_full = smem_u32(&bars->o_full[t]);
    const uint32_t p_half = smem_u32(&bars->p_half[t]), p_full = smem_u32(&bars->p_full[t]);
    uint32_t cons = 0, qc = 0, pc = 0, hc = 0, fc = 0;
    bool any_s = false;              // an S was issued before (its S_t must be free first)
    bool ok = true;
    Cursor cur;

    auto issue_s = [&](int st) -> bool {
        // the softmax warps hold the previous S_t in registers
        if (any_s) {
            if (!warp_wait(s_free, fc & 1, abort_flag)) return false;
            ++fc;
            tc_fence_after();
        }
        any_s = true;
        const uint32_t b = k_lo + st * 2 * kTileStep;                  // K: first half of the stage
#pragma unroll
        for (int kk = 0; kk < C::QK_STEPS; ++kk) {
            const uint32_t off =
                ((kk * C::KSTEP_BYTES / C::SW) * C::PANEL_BYTES + (kk * C::KSTEP_BYTES) % C::SW) >> 4;
            mma_ss_e<C::FP8>(s_tm, q_lo + off, b + off, kHi, kIdS, kk > 0 ? 1u : 0u);
        }
        tc_commit_e(s_full);
        return true;
    };
    auto issue_pv = [&](int st, bool acc) -> bool {
        const uint32_t b = v_lo + (st * 2 + 1) * kTileStep;            // V: second half of the stage
        constexpr int HK = C::PV_STEPS / 2;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            // P was written by the softmax threads (tcgen05.st): order these
            // MMAs after their fence::before_thread_sync + arrive
            if (!warp_wait(hf ? p_full : p_half, hf ? (pc & 1) : (hc & 1), abort_flag)) return false;
            tc_fence_after();
#pragma unroll
            for (int kx = 0; kx < HK; ++kx) {
                const int kk = hf * HK + kx;
                mma_ts_e<C::FP8>(o_tm, p_tm + kk * (C::MMA_K * C::E / 4), b + ((kk * C::MMA_K * C::SW) >> 4), kHi,
                                 kIdPV, (acc || kk > 0) ? 1u : 0u);
            }
        }
        ++hc;
        ++pc;
        tc_commit_e(pv_done);
        return true;
    };
    auto next_kv = [&](int &st) -> bool {
        st = cons % C::NSTAGE;
        const bool r = warp_wait(smem_u32(&bars->kv_full[st]), (cons / C::NSTAGE) & 1, abort_flag);
        ++cons;
        return r;
    };

    for (int r = 0; ok; ++r) {
        Unit U;
        if (!decode_work<SPLIT, HP, C::FP8 && C::D == 128>(p, unit_of_round(r), cur, U)) break;
        const int n = t ? U.n[1] : U.n[0], j0 = U.j0, jn = U.j1;
        if (j0 >= jn) continue;
        int st;
        if (n > j0) {
            ok = warp_wait(smem_u32(&bars->q_full[t]), qc & 1, abort_flag);
            ++qc;
        }
        if (!ok || !next_kv(st)) { ok = false; break; }         // stage j0: K_j0
        if (n > j0) {
            if (!issue_s(st)) { ok = false; break; }
            if (n == j0 + 1) tc_commit_e(q_empty);
        }
        tc_commit_e(smem_u32(&bars->kv_empty[st]));
        for (int j = j0; j < jn; ++j) {
            if (!next_kv(st)) { ok = false; break; }            // stage j+1: V_j, K_j+1
            const bool act = j < n, more = j + 1 < n;
            if (more) {
                if (!issue_s(st)) { ok = false; break; }
                if (j + 2 == n) tc_commit_e(q_empty);
            }
            if (act) {
                if (!issue_pv(st, j > j0)) { ok = false; break; }
                if (!more) tc_commit_e(o_full);
            }
            tc_commit_e(smem_u32(&bars->kv_empty[st]));
        }
    }
    // no tensor-core operation may be in flight when TMEM is released
    tc_commit_e(smem_u32(&bars->drain));
    mbar_wait_drain(smem_u32(&bars->drain), 0);
}

// ---------------------------------------------------------------------------
// Softmax warpgroups (one thread per query row) and the epilogue
// ---------------------------------------------------------------------------

// This thread's row of S_t on a tile with masked elements (keys at local
// column >= lim get score -inf) and its maximum; the same load-and-reduce
// order as load_s_max below, with the mask applied to the loaded words.
__device__ __forceinline__ float load_s_mask_max(uint32_t s_tm, int lim, float (&s)[kTile]) {
    constexpr uint32_t kNegInf = 0xff800000u;
    uint32_t r0[32], r1[32], r2[32], r3[32];
    tmem_ld32(s_tm, r0);
    tmem_ld32(s_tm + 32, r1);
    tmem_wait_ld(r0);
    tmem_wait_ld(r1);
    tmem_ld32(s_tm + 64, r2);
    tmem_ld32(s_tm + 96, r3);
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        r0[i] = i >= lim ? kNegInf : r0[i];
        r1[i] = 32 + i >= lim ? kNegInf : r1[i];
    }
    float m8[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        m8[k] = max3(__uint_as_float(r0[k]), __uint_as_float(r0[8 + k]), __uint_as_float(r0[16 + k]));
        m8[k] = max3(m8[k], __uint_as_float(r0[24 + k]), __uint_as_float(r1[k]));
        m8[k] = max3(m8[k], __uint_as_float(r1[8 + k]), __uint_as_float(r1[16 + k]));
        m8[k] = fmaxf(m8[k], __uint_as_float(r1[24 + k]));
    }
    float m_lo = max3(max3(m8[0], m8[1], m8[2]), max3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
    tmem_wait_ld_after(r2, m_lo);
    tmem_wait_ld(r3);
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        r2[i] = 64 + i >= lim ? kNegInf : r2[i];
        r3[i] = 96 + i >= lim ? kNegInf : r3[i];
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        m8[k] = max3(__uint_as_float(r2[k]), __uint_as_float(r2[8 + k]), __uint_as_float(r2[16 + k]));
        m8[k] = max3(m8[k], __uint_as_float(r2[24 + k]), __uint_as_float(r3[k]));
        m8[k] = max3(m8[k], __uint_as_float(r3[8 + k]), __uint_as_float(r3[16 + k]));
        m8[k] = fmaxf(m8[k], __uint_as_float(r3[24 + k]));
    }
    const float m_hi = max3(max3(m8[0], m8[1], m8[2]), max3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        s[i] = __uint_as_float(r0[i]);
        s[32 + i] = __uint_as_float(r1[i]);
        s[64 + i] = __uint_as_float(r2[i]);
        s[96 + i] = __uint_as_float(r3[i]);
    }
    return fmaxf(m_lo, m_hi);
}

// This thread's row of S_t and its maximum, for a tile with no masked element:
// the maximum of the first 64 columns is taken while the last 64 load.
__device__ __forceinline__ float load_s_max(uint32_t s_tm, float (&s)[kTile]) {
    uint32_t r0[32], r1[32], r2[32], r3[32];
    tmem_ld32(s_tm, r0);
    tmem_ld32(s_tm + 32, r1);
    tmem_wait_ld(r0);
    tmem_wait_ld(r1);
    tmem_ld32(s_tm + 64, r2);
    tmem_ld32(s_tm + 96, r3);
    float m8[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        m8[k] = max3(__uint_as_float(r0[k]), __uint_as_float(r0[8 + k]), __uint_as_float(r0[16 + k]));
        m8[k] = max3(m8[k], __uint_as_float(r0[24 + k]), __uint_as_float(r1[k]));
        m8[k] = max3(m8[k], __uint_as_float(r1[8 + k]), __uint_as_float(r1[16 + k]));
        m8[k] = fmaxf(m8[k], __uint_as_float(r1[24 + k]));
    }
    float m_lo = max3(max3(m8[0], m8[1], m8[2]), max3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
    tmem_wait_ld_after(r2, m_lo);
    tmem_wait_ld(r3);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        m8[k] = max3(__uint_as_float(r2[k]), __uint_as_float(r2[8 + k]), __uint_as_float(r2[16 + k]));
        m8[k] = max3(m8[k], __uint_as_float(r2[24 + k]), __uint_as_float(r3[k]));
        m8[k] = max3(m8[k], __uint_as_float(r3[8 + k]), __uint_as_float(r3[16 + k]));
        m8[k] = fmaxf(m8[k], __uint_as_float(r3[24 + k]));
    }
    const float m_hi = max3(max3(m8[0], m8[1], m8[2]), max3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        s[i] = __uint_as_float(r0[i]);
        s[32 + i] = __uint_as_float(r1[i]);
        s[64 + i] = __uint_as_float(r2[i]);
        s[96 + i] = __uint_as_float(r3[i]);
    }
    return fmaxf(m_lo, m_hi);
}

// exp2 of 64 scores (one half row) into packed P words: 32 words for 16-bit
// types, 16 for e4m3.  Returns the fp32 sum.
template <class C>
__device__ __forceinline__ float exp_half(const float *x, uint64_t c2, uint64_t nm2, uint32_t *w) {
    uint64_t ls[2] = {0ull, 0ull};
    if constexpr (!C::FP8) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            float a, b;
            unpack_f2(fma_f2(pack_f2(x[2 * i], x[2 * i + 1]), c2, nm2), a, b);
            a = ex2(a);
            b = ex2(b);
            ls[i & 1] = add_f2(ls[i & 1], pack_f2(a, b));
            w[i] = pack2<C::ELEM>(a, b);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float a, b, d, e;
            unpack_f2(fma_f2(pack_f2(x[4 * i], x[4 * i + 1]), c2, nm2), a, b);
            unpack_f2(fma_f2(pack_f2(x[4 * i + 2], x[4 * i + 3]), c2, nm2), d, e);
            a = ex2(a);
            b = ex2(b);
            d = ex2(d);
            e = ex2(e);
            ls[0] = add_f2(ls[0], pack_f2(a, b));
            ls[1] = add_f2(ls[1], pack_f2(d, e));
            w[i] = pack4_e4m3(a, b, d, e);
        }
    }
    float a, b;
    unpack_f2(add_f2(ls[0], ls[1]), a, b);
    return a + b;
}

template <class C>
__device__ __forceinline__ void rescale_o(uint32_t o_tm, float alpha) {
#pragma unroll 1
    for (int ch = 0; ch < C::D / 32; ++ch) {
        uint32_t r[32];
        tmem_ld32(o_tm + 32 * ch, r);
        tmem_wait_ld(r);
#pragma unroll
        for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
        tmem_st32(o_tm + 32 * ch, r);
    }
    tmem_wait_st();
}

// P from scores held in registers, one half row (64 keys) at a time, each
// half published on its own barrier as soon as it is in TMEM: the tensor
// pipe starts PV over the first 64 keys while the second half is computed.
// P words of keys 0-63 land below those of keys 64-127 (32 columns per half
// for 16-bit P, 16 for e4m3).  Returns the fp32 sum.
//
// O_t holds PV_t_{j-1} (complete, since S_t_j was issued after it) and is
// rescaled by alpha when `rescale` is set, before the first half of P_t_j is
// published; that happens after the first half is stored, while only the
// second half of the scores is live.
//
// With separate P buffers (p_tm apart from S), pv_wait != 0 names the barrier
// (bit 31: the phase parity) of the previous PV of this tile, which must be
// done before P_t is overwritten or O_t rescaled; it is waited for after the
// first half of P is computed, just before it is stored.
template <class C>
__device__ __forceinline__ float exp_store_publish(uint32_t p_tm, const float (&s)[kTile], float c, float neg_m,
                                                   bool rescale, uint32_t o_tm, float alpha, uint32_t half_bar,
                                                   uint32_t full_bar, int lane, uint32_t pv_wait = 0,
                                                   volatile int *abort_flag = nullptr) {
    const uint64_t c2 = pack_f2(c, c), nm2 = pack_f2(neg_m, neg_m);
    float sum = 0.f;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        if constexpr (!C::FP8) {
            uint32_t w[32];
            sum += exp_half<C>(s + 64 * h, c2, nm2, w);
            if (h == 0 && pv_wait != 0) {
                if (warp_wait_inline(pv_wait & 0x7fffffffu, pv_wait >> 31, abort_flag)) tc_fence_after();
                else rescale = false;            // aborted: the caller sees the abort flag
            }
            tmem_st32(p_tm + 32 * h, w);
        } else {
            uint32_t w[16];
            sum += exp_half<C>(s + 64 * h, c2, nm2, w);
            if (h == 0 && pv_wait != 0) {
                if (warp_wait_inline(pv_wait & 0x7fffffffu, pv_wait >> 31, abort_flag)) tc_fence_after();
                else rescale = false;
            }
            tmem_st16(p_tm + 16 * h, w);
        }
        if (h == 0 && rescale) rescale_o<C>(o_tm, alpha);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(h ? full_bar : half_bar);
    }
    return sum;
}

template <class C>
__device__ __forceinline__ void store_chunk(uint8_t *dst, const uint32_t (&r)[32], float inv) {
    if constexpr (C::FP8) {
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            w[i] = pack4_e4m3(__uint_as_float(r[4 * i]) * inv, __uint_as_float(r[4 * i + 1]) * inv,
                              __uint_as_float(r[4 * i + 2]) * inv, __uint_as_float(r[4 * i + 3]) * inv);
        uint4 *d4 = reinterpret_cast<uint4 *>(dst);
        d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
        d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
    } else {
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
            w[i] = pack2<C::ELEM>(__uint_as_float(r[2 * i]) * inv, __uint_as_float(r[2 * i + 1]) * inv);
        uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
        for (int i = 0; i < 4; ++i) d4[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
    }
}

// 32 values of O (one TMEM chunk) in the output type into row `row` of a
// warp's staging panel (SW bytes per row, the TMA swizzle: 16-byte chunk c
// of a row goes to c ^ (row % 8) for 128-byte rows, ^ (row / 2) % 4 for 64,
// ^ (row / 4) % 2 for 32), starting at byte `col_bytes` of the row.
template <class C>
__device__ __forceinline__ void stage_chunk(uint8_t *stg_row, int row, int col_bytes, const uint32_t (&r)[32],
                                            float inv) {
    const int swz = C::SW == 128 ? (row & 7) : C::SW == 64 ? ((row >> 1) & 3) : ((row >> 2) & 1);
    const int c0 = col_bytes >> 4;
    if constexpr (C::FP8) {
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            w[i] = pack4_e4m3(__uint_as_float(r[4 * i]) * inv, __uint_as_float(r[4 * i + 1]) * inv,
                              __uint_as_float(r[4 * i + 2]) * inv, __uint_as_float(r[4 * i + 3]) * inv);
#pragma unroll
        for (int i = 0; i < 2; ++i)
            *reinterpret_cast<uint4 *>(stg_row + (((c0 + i) ^ swz) << 4)) =
                make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
    } else {
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
            w[i] = pack2<C::ELEM>(__uint_as_float(r[2 * i]) * inv, __uint_as_float(r[2 * i + 1]) * inv);
#pragma unroll
        for (int i = 0; i < 4; ++i)
            *reinterpret_cast<uint4 *>(stg_row + (((c0 + i) ^ swz) << 4)) =
                make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
    }
}

template <class C, bool SPLIT, bool HP>
__device__ void softmax_wg(const Params &p, Bars *bars, uint32_t tmem, int warp, int lane, const CUtensorMap *tmO,
                           uint8_t *stg) {
    volatile int *abort_flag = &bars->abort;
    const int t = warp >> 2, wq = warp & 3;
    const uint32_t lane_base = tmem + ((uint32_t)(wq * 32) << 16);
    const uint32_t s_tm = lane_base + (t ? C::S_COL1 : C::S_COL0);
    const uint32_t o_tm = lane_base + (t ? C::O_COL1 : C::O_COL0);
    const uint32_t p_tm = lane_base + (t ? C::P_COL1 : C::P_COL0);      // = s_tm unless PSEP
    const uint32_t s_bar = smem_u32(&bars->s_full[t]);
    const uint32_t sf_bar = smem_u32(&bars->s_free[t]), pv_bar = smem_u32(&bars->pv_done[t]);
    uint32_t pvc = 0;                          // PSEP: PVs of this tile published so far
    const uint32_t ph_bar = smem_u32(&bars->p_half[t]);
    const uint32_t p_bar = smem_u32(&bars->p_full[t]);
    const uint32_t o_bar = smem_u32(&bars->o_full[t]);
    const float c = p.scale * kLog2e;          // scores in log2 units: s * scale * log2(e)
    const bool causal = p.mask == FMHA_MASK_CAUSAL;
    uint32_t s_ph = 0, o_ph = 0;
    bool ok = true;
    Cursor cur;
    for (int r = 0; ok; ++r) {
        Unit U;
        if (!decode_work<SPLIT, HP, C::FP8 && C::D == 128>(p, unit_of_round(r), cur, U)) break;
        const int n = U.n[t], nu = U.nu[t], j0 = U.j0;
        const int row = tile_row0<HP>(U, t) + wq * 32 + lane;  // query row within the sequence
        // keys [0, key_end) are visible to this row
        int key_end = U.sk;
        if (causal) key_end = imin(key_end, row + 1 + (p.causal_type == FMHA_CAUSAL_QEND ? U.sk - U.sq : 0));
        float m_ref = -INFINITY;   // reference max (log2 units) that P and O are relative to
        float l = 0.f;             // running sum of P
        for (int j = j0; j < n; ++j) {
            if (!warp_wait(s_bar, s_ph, abort_flag)) { ok = false; break; }
            s_ph ^= 1;
            tc_fence_after();
            float s[kTile];
            float m_raw;
            if (j >= nu) {                                   // boundary tile
                m_raw = load_s_mask_max(s_tm, key_end - j * kTile, s);
            } else {
                m_raw = load_s_max(s_tm, s);
            }
            if constexpr (C::PSEP) {
                // S_t is in registers: the next S may overwrite it.  Every
                // thread arrives on its own (a lane-0 arrive after a warp
                // sync made the compiler spill the live scores)
                tc_fence_before();
                mbar_arrive(sf_bar);
            }
            const float m_tile = m_raw * c;                  // scale > 0 keeps the argmax
            const bool resc = m_tile > m_ref + kRescaleLog2;
            float alpha = 1.f;
            if (resc) {
                alpha = ex2(m_ref - m_tile);                 // 0 when m_ref = -inf
                l *= alpha;
                m_ref = m_tile;
            }
            if constexpr (C::PSEP) {
                // P_t and O_t are free once this tile's previous PV is done
                l += exp_store_publish<C>(p_tm, s, c, m_ref == -INFINITY ? 0.f : -m_ref,
                                          j > j0 && __any_sync(0xffffffffu, resc), o_tm, alpha, ph_bar, p_bar,
                                          lane, pvc > 0 ? (pv_bar | (((pvc - 1) & 1u) << 31)) : 0u, abort_flag);
                ++pvc;
                if (*abort_flag) { ok = false; break; }
            } else {
                l += exp_store_publish<C>(s_tm, s, c, m_ref == -INFINITY ? 0.f : -m_ref,
                                          j > j0 && __any_sync(0xffffffffu, resc), o_tm, alpha, ph_bar, p_bar, lane);
            }
        }
        if (!ok) break;

        // epilogue: O = out_scale * O_acc / l, cast, store; LSE = ln(sum exp(scale s))
        const bool have = n > j0;
        if (have) {
            if (!warp_wait(o_bar, o_ph, abort_flag)) { ok = false; break; }
            o_ph ^= 1;
            tc_fence_after();
        }
        const bool valid = row < U.sq;
        const int qh = tile_head<HP>(U, t);                    // query head of this tile
        if constexpr (SPLIT) {
            // split-KV: normalised fp32 partial O and its LSE for the combine
            const int64_t prow = ((int64_t)U.split * p.part_rows + U.q_row + row) * p.H + qh;
            float *po = p.part_o + prow * C::D;
            const float pinv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
            for (int ch = 0; ch < C::D / 32; ++ch) {
                uint32_t r[32];
                if (have) {
                    tmem_ld32(o_tm + 32 * ch, r);
                    tmem_wait_ld(r);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) r[i] = 0u;
                }
                if (valid) {
                    float4 *d4 = reinterpret_cast<float4 *>(po + 32 * ch);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        d4[i] = make_float4(__uint_as_float(r[4 * i]) * pinv, __uint_as_float(r[4 * i + 1]) * pinv,
                                            __uint_as_float(r[4 * i + 2]) * pinv, __uint_as_float(r[4 * i + 3]) * pinv);
                }
            }
            if (valid) p.part_lse[prow] = l > 0.f ? (m_ref + log2f(l)) * kLn2 : -INFINITY;
            continue;
        }
        const float inv = l > 0.f ? p.out_scale / l : 0.f;
        // this warp's 32 rows go out through shared memory and a TMA store
        // (whole 128-byte lines) when they all belong to this sequence; rows
        // past a fixed-length sequence's end fall outside the tensor map and
        // are not written.  A packed (varlen) warp that crosses its
        // sequence's end stores its rows one by one.
        const int wrow0 = tile_row0<HP>(U, t) + wq * 32;
        const bool by_tma = wrow0 < U.sq && (!p.varlen || wrow0 + 32 <= U.sq);
        if (by_tma) {
            uint8_t *srow = stg + warp * C::STG_WARP + lane * C::SW;
            constexpr int CH_PER_PANEL = C::BOX_D / 32;
#pragma unroll 1
            for (int pn = 0; pn < C::PANELS; ++pn) {
                // the warp's previous store has read the staging panel
                if (lane == 0) bulk_wait_read();
                __syncwarp();
#pragma unroll 1
                for (int c2 = 0; c2 < CH_PER_PANEL; ++c2) {
                    uint32_t r[32];
                    if (have) {
                        tmem_ld32(o_tm + 32 * (pn * CH_PER_PANEL + c2), r);
                        tmem_wait_ld(r);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) r[i] = 0u;
                    }
                    stage_chunk<C>(srow, lane, c2 * 32 * C::E, r, inv);
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) {
                    const uint32_t src = smem_u32(stg + warp * C::STG_WARP);
                    if (p.varlen) tma_store_3d(tmO, src, pn * C::BOX_D, qh, U.q_row + wrow0);
                    else tma_store_4d(tmO, src, pn * C::BOX_D, qh, wrow0, U.b);
                    bulk_commit();
                }
            }
        } else {
            uint8_t *orow = reinterpret_cast<uint8_t *>(p.o) +
                            (((int64_t)U.q_row + row) * p.H + qh) * (int64_t)(C::D * C::E);
#pragma unroll 1
            for (int ch = 0; ch < C::D / 32; ++ch) {
                uint32_t r[32];
                if (have) {
                    tmem_ld32(o_tm + 32 * ch, r);
                    tmem_wait_ld(r);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) r[i] = 0u;
                }
                if (valid) store_chunk<C>(orow + ch * 32 * C::E, r, inv);
            }
        }
        if (valid && p.lse) {
            const int64_t li = p.varlen ? (int64_t)qh * p.total_length + U.q_row + row
                                        : ((int64_t)U.b * p.H + qh) * p.Sq + row;
            p.lse[li] = l > 0.f ? (m_ref + log2f(l)) * kLn2 : -INFINITY;
        }
    }
    // the CTA's shared memory must outlive the stores that read it
    if (!SPLIT && lane == 0) bulk_wait_all();
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------

template <class C, bool SPLIT, bool HP>
__global__ void __launch_bounds__(kThreads, 1)
    fmha_fwd_sm103_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                          const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                          const Params p) {
    static_assert(C::TURN_AT >= 0 && C::TURN_EARLY >= 0, "the turn hand-over is inside the S group");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *sQ = smem;                               // 2 Q tiles
    uint8_t *sKV = smem + 2 * C::TILE_BYTES;          // NS K/V stages
    uint8_t *sStg = sKV + C::NS * C::TILE_BYTES;      // O staging of the softmax warps
    Bars *bars = reinterpret_cast<Bars *>(sStg + C::STG_BYTES);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int t = 0; t < 2; ++t) {
            mbar_init(smem_u32(&bars->q_full[t]), 1);
            mbar_init(smem_u32(&bars->q_empty[t]), 1);
            mbar_init(smem_u32(&bars->s_full[t]), 1);
            mbar_init(smem_u32(&bars->p_half[t]), 4);   // one arrival per softmax warp
            mbar_init(smem_u32(&bars->p_full[t]), 4);
            mbar_init(smem_u32(&bars->o_full[t]), 1);
        }
        mbar_init(smem_u32(&bars->drain), 2);             // one commit per issuing warp
        for (int t = 0; t < 2; ++t) {
            mbar_init(smem_u32(&bars->s_free[t]), 128);   // one arrival per softmax thread
            mbar_init(smem_u32(&bars->pv_done[t]), 1);
        }
        mbar_init(smem_u32(&bars->turn[0]), 1);
        mbar_init(smem_u32(&bars->turn[1]), 1);
        for (int s = 0; s < C::NSTAGE; ++s) {
            mbar_init(smem_u32(&bars->kv_full[s]), 1);
            mbar_init(smem_u32(&bars->kv_empty[s]), 2);   // released by both issuing warps
        }
        bars->abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        mbar_arrive(smem_u32(&bars->turn[0]));            // tile 0's lane issues first
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(&bars->tmem_base), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    // a dependent kernel (the split-KV combine) may be scheduled as CTAs of
    // this grid exit; it waits for this grid's completion before its reads
    if constexpr (SPLIT) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp < kProducerWarp) {
        softmax_wg<C, SPLIT, HP>(p, bars, tmem, warp, lane, &tmO, sStg);
    } else if (warp == kProducerWarp) {
        if (lane == 0) producer<C, SPLIT, HP>(p, &tmQ, &tmK, &tmV, sQ, sKV, bars);
    } else if constexpr (C::PSEP) {
        mma_issuer_psep<C, SPLIT, HP>(p, sQ, sKV, bars, tmem, warp - kMmaWarp);
    } else {
        mma_issuer<C, SPLIT, HP>(p, sQ, sKV, bars, tmem, warp - kMmaWarp);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) {
        __syncwarp();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// Host side: tensor maps and launch
// ---------------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

int sm_count() {
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

// [rows, heads, D] (varlen, rank 3) or [batch, rows, heads, D] (rank 4) with
// a 128-row box of one head and one swizzle panel of the head dim.
template <class C>
bool encode_map(CUtensorMap *m, const void *base, int heads, int rows, int batch, bool varlen,
                int box_rows = kTile) {
    auto fn = encode_fn();
    if (!fn) return false;
    const CUtensorMapDataType dt = C::ELEM == kBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                   : C::ELEM == kF16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                     : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    const CUtensorMapSwizzle sw = C::SW == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                                  : C::SW == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                : CU_TENSOR_MAP_SWIZZLE_32B;
    const cuuint64_t row_bytes = (cuuint64_t)C::D * C::E;
    cuuint64_t dims[4] = {(cuuint64_t)C::D, (cuuint64_t)heads, (cuuint64_t)imax(rows, 1), (cuuint64_t)batch};
    cuuint64_t strides[3] = {row_bytes, row_bytes * heads, row_bytes * heads * (cuuint64_t)imax(rows, 1)};
    cuuint32_t box[4] = {(cuuint32_t)C::BOX_D, 1, (cuuint32_t)box_rows, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUresult r = fn(m, dt, varlen ? 3 : 4, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <class C>
int launch_cfg(const Params &p, cudaStream_t stream) {
    CUtensorMap tq, tk, tv, to;
    const int rq = p.varlen ? (int)p.total_length : p.Sq;
    const int rk = p.varlen ? (int)p.total_length : p.Sk;
    const int nb = p.varlen ? 1 : p.B;
    if (!encode_map<C>(&tq, p.q, p.H, rq, nb, p.varlen) || !encode_map<C>(&tk, p.k, p.H_k, rk, nb, p.varlen) ||
        !encode_map<C>(&tv, p.v, p.H_k, rk, nb, p.varlen))
        return FMHA_ERR_CUDA;
    // O: the epilogue's TMA stores, 32 rows (one softmax warp) per box; the
    // split-KV instantiation writes fp32 partials instead and never uses it
    if (!encode_map<C>(&to, p.part_o ? p.q : p.o, p.H, rq, nb, p.varlen, 32)) return FMHA_ERR_CUDA;
    const int nsm = sm_count();
    if (nsm <= 0) return FMHA_ERR_CUDA;
    int64_t units;
    if (p.varlen)
        units = (int64_t)p.H * (p.B + p.total_length / kUnitRows + 1);   // upper bound
    else
        units = (int64_t)p.B * p.H * ((p.Sq + kUnitRows - 1) / kUnitRows);
    // head pairs: instantiated for D = 128 (the head dim of the split-KV and
    // short-query workloads); other head dims keep one head per unit
    const bool hp = C::D == 128 && p.hpair;
    if (hp) units = (int64_t)p.B * (p.H / 2);
    units *= p.num_splits;
    const int grid = (int)(units < nsm ? units : nsm);
    if (grid <= 0) return FMHA_OK;
    // split-KV is a separate instantiation so the plain kernel keeps its code
    void (*kern)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, Params) =
        p.part_o ? fmha_fwd_sm103_kernel<C, true, false> : fmha_fwd_sm103_kernel<C, false, false>;
    if constexpr (C::D == 128)
        if (hp) kern = p.part_o ? fmha_fwd_sm103_kernel<C, true, true> : fmha_fwd_sm103_kernel<C, false, true>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES) != cudaSuccess) {
        cudaGetLastError();
        return FMHA_ERR_CUDA;
    }
    kern<<<grid, kThreads, C::SMEM_BYTES, stream>>>(tq, tk, tv, to, p);
    if (cudaGetLastError() != cudaSuccess) return FMHA_ERR_CUDA;
    return FMHA_OK;
}

template <int D>
int launch_d(const Params &p, cudaStream_t stream) {
    switch (p.dtype) {
    case FMHA_BF16: return launch_cfg<Cfg<D, kBF16>>(p, stream);
    case FMHA_F16: return launch_cfg<Cfg<D, kF16>>(p, stream);
    case FMHA_E4M3: return launch_cfg<Cfg<D, kE4M3>>(p, stream);
    default: return FMHA_ERR_INVALID_ARG;
    }
}

}  // namespace

int launch_sm103(const Params &p, cudaStream_t stream) {
    switch (p.D) {
    case 32: return launch_d<32>(p, stream);
    case 64: return launch_d<64>(p, stream);
    case 128: return launch_d<128>(p, stream);
    default: return FMHA_ERR_INVALID_ARG;
    }
}

int sm103_set_wait_limit(unsigned long long ns) {
    const unsigned long long v = ns ? ns : kTimeoutNs;
    if (cudaMemcpyToSymbol(g_wait_ns, &v, sizeof(v)) != cudaSuccess) {
        cudaGetLastError();
        return FMHA_ERR_CUDA;
    }
    return FMHA_OK;
}

int sm103_set_test_gate(int on) {
    const int v = on ? 1 : 0;
    if (cudaMemcpyToSymbol(g_test_gate, &v, sizeof(v)) != cudaSuccess) {
        cudaGetLastError();
        return FMHA_ERR_CUDA;
    }
    return FMHA_OK;
}

int sm103_read_status(int reset) {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_status, sizeof(int)) != cudaSuccess) {
        cudaGetLastError();
        return FMHA_ERR_CUDA;
    }
    if (reset) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_status, &zero, sizeof(int)) != cudaSuccess) {
            cudaGetLastError();
            return FMHA_ERR_CUDA;
        }
    }
    return v;
}

}  // namespace fmha
