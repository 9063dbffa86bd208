// Tensor-core (tcgen05 / TMEM) kernels of the MTTKRP path on sm_103a, all
// fp32-accurate: every operand is split into two low-precision terms whose
// cross products the tensor cores accumulate in fp32, so the result matches an
// fp32 contraction to within a few fp32 roundings of the sum of magnitudes.
//
// Common structure.  A CTA owns a 128 x BN tile of M_k (rows i, columns r) and
// a contiguous range of pre indices pi; for every pi the contraction over the
// inner-group index j runs in K-steps.  A TMA warp brings tiles of Y_(k)
// (tensor maps over the natural layout of Y, or over its fp16 images) into a
// ring of shared-memory stages, one elected thread issues tcgen05.mma into a
// double-buffered TMEM accumulator, and epilogue warps drain it with
// tcgen05.ld after a bounded number of K-steps (TMEM accumulation truncates),
// scale each column by the pre-mode factor product G(pi, r) and add it into
// fp32 registers.  Every mbarrier wait is bounded in time; on expiry the
// kernel records an error word, stops issuing, waits (bounded) for its own
// copies and MMAs and frees its TMEM before returning.
//
// The main kernels:
//  * tc_img_kernel: kind::f16 on a two-term fp16 split of Y (hi and lo images
//    written once per call, with a power-of-two scale per slab of mode 0) and
//    of the inner Khatri-Rao rows; products hi*hi + hi*lo + lo*hi.  Modes
//    other than the innermost read K-major images; the innermost one reads its
//    natural (i-fastest) image directly as an MN-major A operand, or a
//    transposed image where the MN-major form does not apply.  A SMALL form
//    stacks several pre indices in one tile for short inner groups.
//  * tc_h2_kernel: the same split formed in TMEM by producer warps from raw
//    fp32 tiles (large R; register split between warpgroups).
//  * tc_mttkrp_kernel: kind::tf32, 3xTF32 split (raw fp32 tile as hi,
//    producer warps write lo = y - tf32(y)); K-major and innermost forms.
//  * tc_tmem_kernel: the 3xTF32 kernel with A in TMEM, for large R on the
//    innermost mode.
// Helpers: the per-slab max|Y| pass and the fp16 image splits of Y (natural
// and transposed), the pre-swizzled B images of the inner Khatri-Rao table
// (tf32 and fp16, with per-column scales), the explicit Khatri-Rao image
// builder, the mode-n-product operand preparation, and the tensor-pipe
// throughput probe.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <atomic>
#include <cstdio>
#include <cstring>

#include "scale.cuh"
#include "tc.h"

namespace mk {

// Error word set by kernels whose bounded waits expire (read by the host
// through mttkrp_device_status).
__device__ uint32_t g_device_status = 0;

namespace {

constexpr int kBM = 128;
constexpr int kBK = 16;           // contraction indices per K-step (64-byte rows)
constexpr int kChunkSteps = 8;    // at most this many K-steps accumulate in TMEM between drains
constexpr int kEpiWarps = 16;  // 4 per TMEM lane quadrant
// Warp roles: 0 TMA, 1 MMA, then the operand-producer warps, then the epilogue.
template <bool INNER>
struct Roles {
    static constexpr int kProdWarps = 2;
    static constexpr int kProdThreads = kProdWarps * 32;
    static constexpr int kFirstEpi = 2 + kProdWarps;
    static constexpr int kThreads = (kFirstEpi + kEpiWarps) * 32;
};

constexpr unsigned long long kWaitNs = 1000000000ull;  // 1 s bound on every wait
constexpr uint32_t kTf32Mask = 0xFFFFE000u;

// status codes (bit flags)
constexpr uint32_t kStatusTimeoutTma = 1u << 0;
constexpr uint32_t kStatusTimeoutLo = 1u << 1;
constexpr uint32_t kStatusTimeoutMma = 1u << 2;
constexpr uint32_t kStatusTimeoutEpi = 1u << 3;
constexpr uint32_t kStatusTimeoutDrain = 1u << 4;

enum Role { kRoleJq = 0, kRoleI = 1, kRoleJp = 2, kRolePP = 3, kRolePQ = 4, kRoles = 5 };

struct TcArgs {
    CUtensorMap ymap;
    CUtensorMap ymap_lo;      // fp16-image kernel: the lo image (ymap holds the hi image)
    int rank;                 // tensor-map rank (2..5)
    int slot[kRoles];         // coordinate slot of each role, -1 if absent
    const float* bimg;        // B images [n-tile][K-step][hi|lo][BN rows x 64 B]
    const float* gtab;        // npre x R
    float* dst;
    int64_t dst_split_stride;
    int64_t I, R;
    int64_t npre, pre_per_split;
    int64_t nQ;               // size of the merged q-side pre dimension
    int KS;                   // K-steps per pi
    int jq_steps;             // K-steps per value of jp (K-contiguous variant)
    int withhold_signal;      // test hook: skip the first accumulator-ready commit
    int jc_per_split;         // > 0: blockIdx.z splits the B chunks (this many a CTA), every
                              // CTA takes all pre indices (explicit Khatri-Rao product)
    int64_t ttm_q;            // > 0: mode-n product; tile row m is (p, q) = (m / ttm_q, m % ttm_q)
                              // of X viewed [P, N, Q], and column j goes to T[p, j, q]
    int64_t tiles_y;          // > 0 (image kernel, not stacked): row tiles, taken by the CTAs of
                              // one grid column in turn (blockIdx.y, + gridDim.y, ...); 0: one
                              // row tile a CTA, blockIdx.y
    uint32_t y_box_bytes;     // bytes of one Y tile copy
    // small-I variant: ps pre indices share one 128-row tile (rows slot * I + i)
    int ps;                   // pre-index slots per tile (1 otherwise)
    int64_t batch_len;        // slots never cross a multiple of this pre index
    // two-term fp16 split only
    const uint32_t* ymax_bits;   // max |Y| as fp32 bits (device)
    const uint32_t* slab_bits;   // max |Y| of every slab of mode 0 (one slab: the whole tensor)
    int64_t slab_div;            // pre indices a slab (slab of pi = pi / slab_div)
    int slab_rows;               // 1: the slab is the output row (mode 0, per-slab scales)
    const float* colscale;       // power-of-two scale of each Binner column (R)
    uint32_t* status;
    // image kernel converting in place (mode 0, the first mode of a call): fp32
    // Y tiles (yfmap: two 32-index boxes a K-step; ymap and ymap_lo then map the
    // images it stores); the out-of-range flag the conversion sets
    CUtensorMap yfmap;
    uint32_t* ovf;
    // non-null: the kernel runs only if *enable is set (the exact redo after a
    // converting launch whose sampled scales were too small)
    const uint32_t* enable;
    int g_ones;               // every G entry is 1 (mode-n product): the epilogue adds Z as is
};

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ unsigned long long gtimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ uint32_t mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok;
}

// Blocking probe: the thread is suspended (no issue slots used) until the phase
// completes or about kSuspendNs elapse.
constexpr uint32_t kSuspendNs = 20000;

__device__ __forceinline__ uint32_t mbar_try_wait_suspend(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendNs)
        : "memory");
    return ok;
}

// Non-blocking test of a phase (returns at once).
__device__ __forceinline__ uint32_t mbar_test_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok;
}

// Slow path of wait_bounded: suspend-and-retry until the phase completes, the
// CTA is aborted, or kWaitNs pass (then the CTA is aborted and `code` recorded).
// The clock is first read after one suspension has run out without the phase
// completing, so a wait that ends within the first suspension (the common case)
// costs no timer read; the bound is kWaitNs plus one suspension.
__device__ __forceinline__ bool wait_slow_body(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                               uint32_t* status, uint32_t code) {
    unsigned long long t0 = 0;
    bool timing = false;
    while (true) {
        if (mbar_try_wait_suspend(bar, parity)) return true;
        if (*abort_flag) return false;
        if (!timing) {
            t0 = gtimer();
            timing = true;
        } else if (gtimer() - t0 > kWaitNs) {
            *abort_flag = 1;
            atomicOr(status, code);
            return false;
        }
    }
}
__device__ __noinline__ bool wait_slow(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                       uint32_t* status, uint32_t code) {
    return wait_slow_body(bar, parity, abort_flag, status, code);
}

// Wait for the phase of `bar` with the given parity; false if the CTA was
// aborted or the wait exceeded kWaitNs.
__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                             uint32_t* status, uint32_t code) {
    if (mbar_try_wait(bar, parity)) return true;
    return wait_slow(bar, parity, abort_flag, status, code);
}

// Like wait_bounded but ignores the abort flag (used to drain in-flight work).
__device__ __forceinline__ bool wait_drain_body(uint64_t* bar, uint32_t parity, uint32_t* status) {
    unsigned long long t0 = 0;
    bool timing = false;
    while (!mbar_try_wait_suspend(bar, parity)) {
        if (!timing) {
            t0 = gtimer();
            timing = true;
        } else if (gtimer() - t0 > kWaitNs) {
            atomicOr(status, kStatusTimeoutDrain);
            return false;
        }
    }
    return true;
}
__device__ __noinline__ bool wait_drain(uint64_t* bar, uint32_t parity, uint32_t* status) {
    return wait_drain_body(bar, parity, status);
}

// Fully inlined forms for kernels that change their register allotment with
// setmaxnreg: ptxas cannot allocate registers around calls in such kernels.
__device__ __forceinline__ bool wait_bounded_inl(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                                 uint32_t* status, uint32_t code) {
    if (mbar_try_wait(bar, parity)) return true;
    return wait_slow_body(bar, parity, abort_flag, status, code);
}
__device__ __forceinline__ bool wait_drain_inl(uint64_t* bar, uint32_t parity, uint32_t* status) {
    return wait_drain_body(bar, parity, status);
}

__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// TMA box coordinates from the role values: c[p] = role[r] for slot[r] == p,
// 0 where no role maps (static indexing only, so everything stays in registers)
__device__ __forceinline__ void tma_coords(const int* slot, const int* role, int* c) {
#pragma unroll
    for (int p = 0; p < 5; ++p) {
        int v = 0;
#pragma unroll
        for (int r = 0; r < kRoles; ++r) v = slot[r] == p ? role[r] : v;
        c[p] = v;
    }
}

__device__ __forceinline__ void tma_load(const CUtensorMap* map, int rank, const int* c, void* dst,
                                         uint64_t* bar) {
    const uint64_t m = reinterpret_cast<uint64_t>(map);
    const uint32_t d = smem_u32(dst), b = smem_u32(bar);
    switch (rank) {
        case 2:
            asm volatile(
                "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                " [%0], [%1, {%2, %3}], [%4];" ::"r"(d),
                "l"(m), "r"(c[0]), "r"(c[1]), "r"(b)
                : "memory");
            break;
        case 3:
            asm volatile(
                "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(d),
                "l"(m), "r"(c[0]), "r"(c[1]), "r"(c[2]), "r"(b)
                : "memory");
            break;
        case 4:
            asm volatile(
                "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(d),
                "l"(m), "r"(c[0]), "r"(c[1]), "r"(c[2]), "r"(c[3]), "r"(b)
                : "memory");
            break;
        default:
            asm volatile(
                "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(d),
                "l"(m), "r"(c[0]), "r"(c[1]), "r"(c[2]), "r"(c[3]), "r"(c[4]), "r"(b)
                : "memory");
            break;
    }
}

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Tensor store of one box from shared memory (bulk-group completion): the
// shared-memory writes it reads are fenced to the async proxy first; the group
// is committed, and its reads waited for before the buffer is written again.
__device__ __forceinline__ void tma_store(const CUtensorMap* map, int rank, const int* c, const void* src) {
    const uint64_t m = reinterpret_cast<uint64_t>(map);
    const uint32_t sa = smem_u32(src);
    switch (rank) {
        case 2:
            asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(m),
                         "r"(sa), "r"(c[0]), "r"(c[1])
                         : "memory");
            break;
        case 3:
            asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(m),
                         "r"(sa), "r"(c[0]), "r"(c[1]), "r"(c[2])
                         : "memory");
            break;
        case 4:
            asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
                             m),
                         "r"(sa), "r"(c[0]), "r"(c[1]), "r"(c[2]), "r"(c[3])
                         : "memory");
            break;
        default:
            asm volatile(
                "cp.async.bulk.tensor.5d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5, %6}], [%1];" ::"l"(m),
                "r"(sa), "r"(c[0]), "r"(c[1]), "r"(c[2]), "r"(c[3]), "r"(c[4])
                : "memory");
            break;
    }
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ float4 lds128(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}
__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}
// largest magnitude of two values, NaN if either is NaN
__device__ __forceinline__ float absmax_nan(float a, float b) {
    float d;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(fabsf(a)), "f"(fabsf(b)));
    return d;
}

// K-major, 64-byte swizzle shared-memory matrix descriptor: 8-row groups of
// 64-byte rows, 512 bytes apart.  Everything but the start-address field is
// constant (kDescSw64Hi holds those fields).
constexpr uint64_t kDescSw64Hi = ((uint64_t)1 << 16)           // leading byte offset (unused)
                               | ((uint64_t)(512 >> 4) << 32)  // stride byte offset: 8 rows x 64 B
                               | ((uint64_t)1 << 46)           // descriptor version
                               | ((uint64_t)4 << 61);          // 64-byte swizzle

// Low 32 bits of the descriptor above (start address and leading byte offset);
// the high word is the constant kDescSw64Hi >> 32.
__device__ __forceinline__ uint32_t sdesc_lo(uint32_t saddr) {
    return (uint32_t)kDescSw64Hi | ((saddr & 0x3FFFFu) >> 4);
}

// D (+)= A * B, kind::tf32; a and b are descriptor low words (high word constant)
__device__ __forceinline__ void mma_tf32_w(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo, uint32_t idesc,
                                           uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t.reg .b64 da, db;\n\t"
        "mov.b64 da, {%1, %3};\n\t"
        "mov.b64 db, {%2, %3};\n\t"
        "setp.ne.b32 p, %5, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], da, db, %4, p;\n\t}\n" ::"r"(d_tmem),
        "r"(a_lo), "r"(b_lo), "r"((uint32_t)(kDescSw64Hi >> 32)), "r"(idesc), "r"(acc));
}

// As mma_tf32_w, issued only by the lane whose `leader` is nonzero (the warp runs
// the issue loop together, so its values stay warp-uniform)
__device__ __forceinline__ void mma_tf32_wl(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo, uint32_t idesc,
                                            uint32_t acc, uint32_t leader) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t.reg .b64 da, db;\n\t"
        "mov.b64 da, {%1, %3};\n\t"
        "mov.b64 db, {%2, %3};\n\t"
        "setp.ne.b32 p, %5, 0;\n\t"
        "setp.ne.b32 e, %6, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], da, db, %4, p;\n\t}\n" ::"r"(d_tmem),
        "r"(a_lo), "r"(b_lo), "r"((uint32_t)(kDescSw64Hi >> 32)), "r"(idesc), "r"(acc), "r"(leader));
}

// commit by the lane whose `leader` is nonzero (the lane that issued the MMAs)
__device__ __forceinline__ void mma_commit_l(uint64_t* bar, uint32_t leader) {
    asm volatile(
        "{\n\t.reg .pred e;\n\tsetp.ne.b32 e, %1, 0;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}\n" ::"r"(
            smem_u32(bar)),
        "r"(leader)
        : "memory");
}

// arrive on `bar` once all previously issued MMAs of this thread have completed
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld4(uint32_t taddr, uint32_t* r) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t* r) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

// N consecutive TMEM columns of the warp's 32 lanes (one register per column)
template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t* r) {
    if constexpr (N == 32) {
        tmem_ld32(taddr, r);
    } else if constexpr (N == 16) {
        tmem_ld16(taddr, r);
    } else {
        static_assert(N == 8, "8, 16 or 32 columns");
        tmem_ld8(taddr, r);
    }
}

__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 16 consecutive TMEM columns of the warp's 32 lanes (one register per column)
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

// 8 consecutive TMEM columns of the warp's 32 lanes
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t* r) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// D (+)= A * B, kind::tf32, A (M=128 rows = lanes, 8 columns of K) in tensor
// memory, B by descriptor low word (high word constant)
__device__ __forceinline__ void mma_tf32_ta(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t idesc,
                                            uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t.reg .b64 db;\n\t"
        "mov.b64 db, {%2, %3};\n\t"
        "setp.ne.b32 p, %5, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], db, %4, p;\n\t}\n" ::"r"(d_tmem),
        "r"(a_tmem), "r"(b_lo), "r"((uint32_t)(kDescSw64Hi >> 32)), "r"(idesc), "r"(acc));
}

__device__ __forceinline__ float tf32_lo(float x) {
    return x - __uint_as_float(__float_as_uint(x) & kTf32Mask);
}

// byte offset of (row, k) in a K-major 64-byte-swizzled tile (16 fp32 per row)
__device__ __forceinline__ uint32_t sw64_off(uint32_t row, uint32_t chunk) {
    return row * 64u + (((chunk ^ (row >> 1)) & 3u) << 4);
}

// ---------------------------------------------------------------------------
// 3xTF32 kernel
// ---------------------------------------------------------------------------
//
// Per K-step of 16 indices: a TMA tensor copy brings the 128 x 16 tile of
// Y_(k) (K-major, 64-byte swizzle; for the innermost mode it arrives i-major
// and the producer warps transpose it), one bulk copy brings the matching
// pre-swizzled BN x 16 hi and lo images of the inner Khatri-Rao table, the
// producer warps write lo(y) = y - tf32(y) next to the raw tile, and one
// thread issues per 8-wide k-slice hi*hi + hi*lo + lo*hi (the tensor cores
// read fp32 as tf32 by truncation, so the raw tile is its own hi part).  The
// accumulator is drained after at most 8 K-steps (48 MMAs) while the MMAs
// continue into the second TMEM buffer.
//
// Order of work in a CTA: the inner index range is cut into B-chunks of CK
// K-steps whose hi|lo images stay resident in shared memory; for each chunk the
// CTA walks all of its pi, streaming only Y tiles.  TMEM is drained after every
// "unit" of at most kChunkSteps K-steps of one (chunk, pi) pair.


// 3xTF32 kernel parameters: operand stages (K-major, innermost), resident
// B-chunk kilobytes, TMEM columns per epilogue load, and the ranks from which
// the fp16 split in tensor memory and the tf32 kernel with A in tensor memory
// take over
constexpr int kStages = 5, kStagesInner = 3;
constexpr int kBResKB = 128, kBResInnerKB = 128;
constexpr int kEpiLd = 8;
constexpr int kH2MinR = 160, kTmemMinR = 448;
// TMEM columns per epilogue load of the fp16-split kernels (register-resident
// accumulators in the split-in-TMEM kernel, G-scaled rows in the image kernel)
// and the smallest rank the fp16-image kernel takes
constexpr int kH2EpiLd = 8, kImgEpiLd = 16;
constexpr int kImgMinR = 32;

template <int BN, bool INNER, bool SMALL = false>
struct Smem {
    static constexpr uint32_t kY = kBM * kBK * 4;      // 8 KB: raw Y tile (hi, or i-major staging if INNER)
    static constexpr uint32_t kA = kBM * kBK * 4;      // 8 KB: one K-major A operand tile
    static constexpr uint32_t kB = BN * kBK * 4;       // BN x 64 B, one K-step of B
    static constexpr uint32_t kBRes =
        (uint32_t)(SMALL ? 96 : INNER ? kBResInnerKB : kBResKB) * 1024;  // resident B-chunk
    static constexpr int kCK = (int)(kBRes / (2 * kB));  // K-steps per B-chunk
    // stages: raw Y tile + on-chip operand tile(s); one producer arrival, one
    // MMA wait and one MMA commit per stage
    static constexpr int kRaw = INNER ? kStagesInner : kStages;
    static constexpr int kOps = kRaw;
    static constexpr uint32_t kOp = INNER ? 2 * kA : kA;  // lo (and transposed hi if INNER)
    // per-warp G rows, double-buffered (small-I variant: up to 3 rows per warp)
    static constexpr uint32_t kG = kEpiWarps * 2 * (SMALL ? 3 : 1) * (BN / 4) * 4;
    static constexpr uint32_t kBarBytes = 256;
    static constexpr uint32_t kOffRaw = kBRes;
    static constexpr uint32_t kOffOps = kOffRaw + kRaw * kY;
    static constexpr uint32_t kOffG = kOffOps + kOps * kOp;
    static constexpr uint32_t kOffBars = kOffG + kG;
    static constexpr uint32_t kTotal = 1024 + kOffBars + kBarBytes;
    static_assert(kTotal <= 232448, "shared memory budget");
    static_assert(!SMALL || (uint32_t)(kBM * (BN + 4) * 4) <= kOffG, "slot-reduction buffer must fit");
    static_assert((3 * kRaw + 7) * 8 + 8 <= kBarBytes, "barrier area");
};

// warp-uniform bounded wait: lane 0 waits, the result is broadcast
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          uint32_t* status, uint32_t code) {
    bool ok = true;
    if ((threadIdx.x & 31) == 0) ok = wait_bounded(bar, parity, abort_flag, status, code);
    return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}
__device__ __forceinline__ bool warp_wait_inl(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                              uint32_t* status, uint32_t code) {
    bool ok = true;
    if ((threadIdx.x & 31) == 0) ok = wait_bounded_inl(bar, parity, abort_flag, status, code);
    return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

// Position in a ring of N slots used round-robin: slot, parity of the current
// round, and whether a previous round exists (then the slot must be released
// first, i.e. its "empty" barrier has completed with parity phase ^ 1).
template <int N>
struct Ring {
    int slot = 0;
    uint32_t phase = 0;
    bool reused = false;
    __device__ __forceinline__ void next() {
        if (++slot == N) {
            slot = 0;
            phase ^= 1u;
            reused = true;
        }
    }
};

// This CTA's share of the contraction: a range of pre indices with every B chunk
// (the contraction split over pre indices), or every pre index with a range of
// B chunks (split over chunks: the explicit Khatri-Rao product has one pre
// index).  The host makes every share non-empty.
struct Share {
    int64_t pre_lo, pre_hi;
    int jc0, jc1;
};
__device__ __forceinline__ Share cta_share(const TcArgs& a, int njc) {
    Share s;
    if (a.jc_per_split > 0) {
        s.pre_lo = 0;
        s.pre_hi = a.npre;
        s.jc0 = (int)blockIdx.z * a.jc_per_split;
        s.jc1 = min(njc, s.jc0 + a.jc_per_split);
    } else {
        s.pre_lo = (int64_t)blockIdx.z * a.pre_per_split;
        s.pre_hi = min(a.npre, s.pre_lo + a.pre_per_split);
        s.jc0 = 0;
        s.jc1 = njc;
    }
    return s;
}

template <int BN, bool INNER, bool SMALL>
__global__ void __launch_bounds__(Roles<INNER>::kThreads, 1) tc_mttkrp_kernel(const __grid_constant__ TcArgs a) {
    using L = Smem<BN, INNER, SMALL>;
    using RO = Roles<INNER>;
    constexpr int kPT = RO::kProdThreads;
    constexpr int kFE = RO::kFirstEpi;
    constexpr int CK = L::kCK;
    constexpr int NR = L::kRaw;
    constexpr int NO = L::kOps;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~(uintptr_t)1023);
    uint8_t* bres = smem;
    uint8_t* raw = smem + L::kOffRaw;
    uint8_t* ops = smem + L::kOffOps;
    float* gsm = reinterpret_cast<float*>(smem + L::kOffG);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kOffBars);
    // stage s holds raw Y tile s and operand tile s; K-step t uses stage t % NR
    static_assert(NR == NO, "one operand tile per stage");
    uint64_t* raw_full = bars;                  // [NR] TMA landed
    uint64_t* op_full = raw_full + NR;          // [NR] producers wrote the stage's operand tiles
    uint64_t* stage_empty = op_full + NR;       // [NR] MMAs that read the stage are done
    uint64_t* zfull = stage_empty + NR;         // [2]
    uint64_t* zempty = zfull + 2;               // [2]
    uint64_t* bfull = zempty + 2;               // [1]
    uint64_t* bempty = bfull + 1;               // [1]
    uint64_t* mma_done = bempty + 1;            // [1]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int tid = threadIdx.x;
    const int warp = __shfl_sync(0xffffffffu, tid >> 5, 0);   // warp-uniform
    const int lane = tid & 31;
    const int64_t m0 = (int64_t)blockIdx.y * kBM;
    const int64_t r0 = (int64_t)blockIdx.x * BN;
    const int KS = a.KS;
    const int njc = (KS + CK - 1) / CK;           // B-chunks
    const Share share = cta_share(a, njc);
    const int64_t pre_lo = share.pre_lo, pre_hi = share.pre_hi;
    const int jc0 = share.jc0, jc1 = share.jc1;
    const int64_t npi = pre_hi > pre_lo ? pre_hi - pre_lo : 0;
    auto chunk_len = [&](int jc) { return min(CK, KS - jc * CK); };
    constexpr uint32_t kTmemCols = (2 * BN <= 32) ? 32 : 2 * BN;

    if (tid == 0) {
        for (int s = 0; s < NR; ++s) {
            mbar_init(&raw_full[s], 1);
            mbar_init(&op_full[s], RO::kProdWarps);
            mbar_init(&stage_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&zfull[b], 1);
            mbar_init(&zempty[b], kEpiWarps);
        }
        mbar_init(bfull, 1);
        mbar_init(bempty, 1);
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // Work units: one pre index, or (small-I variant) up to ps consecutive pre
    // indices that share one tile, never crossing a multiple of batch_len.
    auto unit_next = [&](int64_t pi) -> int64_t {
        if (!SMALL) return pi + 1;
        int64_t e = pi + a.ps;
        const int64_t row_end = (pi / a.batch_len + 1) * a.batch_len;
        if (e > row_end) e = row_end;
        return e < pre_hi ? e : pre_hi;
    };
    int64_t nunits = 0;
    if (SMALL) {
        for (int64_t pi = pre_lo; pi < pre_hi; pi = unit_next(pi)) ++nunits;
    } else {
        nunits = npi;
    }
    // K-steps of this CTA: every unit runs the K-steps of the CTA's B chunks
    const int64_t T = nunits * (int64_t)(min(KS, jc1 * CK) - jc0 * CK);

    if (warp == 0) {
        // ------------------------- TMA producer -------------------------
        if (lane == 0) {
            const uint8_t* bimg = reinterpret_cast<const uint8_t*>(a.bimg);
            Ring<NR> rr;
            int64_t issued = 0;
            int jc_loaded = -1;
            bool ok = true;
            // Replace the resident B-chunk with chunk jc once the MMAs of chunk
            // jc - 1 are done.
            auto load_b = [&](int jc) -> bool {
                if (jc > jc0 && !wait_bounded(bempty, (uint32_t)((jc - jc0 - 1) & 1), abort_flag, a.status,
                                            kStatusTimeoutTma))
                    return false;
                const int ck = chunk_len(jc);
                mbar_arrive_expect_tx(bfull, (uint32_t)(ck * 2 * L::kB));
                for (int q = 0; q < ck; ++q) {
                    const int ks = jc * CK + q;
                    const uint8_t* src = bimg + ((int64_t)blockIdx.x * KS + ks) * (int64_t)(2 * L::kB);
                    bulk_load(bres + q * 2 * L::kB, src, 2 * L::kB, bfull);
                }
                jc_loaded = jc;
                return true;
            };
            for (int jc = jc0; jc < jc1 && ok; ++jc) {
                const int ck = chunk_len(jc);
                // The first NR Y tiles of chunk jc only need stages freed by the
                // MMAs of chunk jc - 1, so they are issued before the chunk swap
                // (which waits for those MMAs); later ones need chunk jc's MMAs.
                const int64_t swap_at = issued + NR;
                bool b_pending = true;
                for (int64_t pi = pre_lo; pi < pre_hi && ok; pi = unit_next(pi)) {
                    const int cP = (int)(pi / a.nQ);
                    const int cQ = (int)(pi - (int64_t)cP * a.nQ);
                    for (int q = 0; q < ck; ++q, ++issued, rr.next()) {
                        if (b_pending && issued == swap_at) {
                            b_pending = false;
                            if (!load_b(jc)) {
                                ok = false;
                                break;
                            }
                        }
                        if (rr.reused && !wait_bounded(&stage_empty[rr.slot], rr.phase ^ 1u, abort_flag,
                                                       a.status, kStatusTimeoutTma)) {
                            ok = false;
                            break;
                        }
                        const int ks = jc * CK + q;
                        int role[kRoles];
                        if (INNER) {
                            role[kRoleJq] = ks * kBK;
                            role[kRoleJp] = 0;
                        } else {
                            const int jp = ks / a.jq_steps;
                            role[kRoleJq] = (ks - jp * a.jq_steps) * kBK;
                            role[kRoleJp] = jp;
                        }
                        role[kRoleI] = (int)m0;
                        role[kRolePP] = cP;
                        role[kRolePQ] = cQ;
                        int c[5];
                        tma_coords(a.slot, role, c);
                        mbar_arrive_expect_tx(&raw_full[rr.slot], a.y_box_bytes);
                        tma_load(&a.ymap, a.rank, c, raw + rr.slot * L::kY, &raw_full[rr.slot]);
                    }
                }
                if (ok && b_pending && !load_b(jc)) ok = false;
            }
            // wait (bounded) for copies still in flight before leaving
            for (int64_t u = issued - 1; u >= 0 && u >= issued - NR; --u)
                wait_drain(&raw_full[u % NR], (uint32_t)((u / NR) & 1), a.status);
            if (jc_loaded >= 0) wait_drain(bfull, (uint32_t)((jc_loaded - jc0) & 1), a.status);
        }
    } else if (warp == 1) {
        // ------------------------- MMA issuer -------------------------
        // One thread issues.  Its per-K-step instruction latency bounds the
        // tensor pipe's duty cycle (six MMAs of BN / 2 cycles each per step), so
        // the loop is kept short: one wait and one commit per stage, and the
        // descriptors' low words advance incrementally (high word constant).
        // The whole warp runs the loop (warp-uniform values; lane 0 issues
        // through a predicate): measured faster than lane 0 alone
        constexpr bool kWarpIssue = true;
        const uint32_t leader = lane == 0 ? 1u : 0u;
        auto mma_w = [&](uint32_t d, uint32_t aw, uint32_t bw_, uint32_t idesc_, uint32_t acc) {
            if constexpr (kWarpIssue) mma_tf32_wl(d, aw, bw_, idesc_, acc, leader);
            else mma_tf32_w(d, aw, bw_, idesc_, acc);
        };
        auto commit_w = [&](uint64_t* bar) {
            if constexpr (kWarpIssue) mma_commit_l(bar, leader);
            else mma_commit(bar);
        };
        auto wait_w = [&](uint64_t* bar, uint32_t par) -> bool {
            bool r = wait_bounded(bar, par, abort_flag, a.status, kStatusTimeoutMma);
            if constexpr (kWarpIssue) r = __all_sync(0xffffffffu, r);
            return r;
        };
        if (kWarpIssue || lane == 0) {
            const uint32_t idesc = (1u << 4) | (2u << 7) | (2u << 10) |
                                   ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);
            const uint32_t raw_s = smem_u32(raw);
            const uint32_t ops_s = smem_u32(ops);
            const uint32_t a_hi0 = sdesc_lo(INNER ? ops_s : raw_s);
            const uint32_t a_lo0 = sdesc_lo(INNER ? ops_s + L::kA : ops_s);
            constexpr uint32_t kAhiStep = (INNER ? L::kOp : L::kY) >> 4;
            constexpr uint32_t kAloStep = L::kOp >> 4;
            const uint32_t b_w0 = sdesc_lo(smem_u32(bres));
            constexpr uint32_t kBStep = (2 * L::kB) >> 4;   // one K-step of the B-chunk
            constexpr uint32_t kBLo = L::kB >> 4;           // lo image after the hi image
            int slot = 0;
            uint32_t phase = 0;
            uint32_t ahi = a_hi0, alo = a_lo0;
            int zb = 0;          // TMEM buffer of the current unit
            uint32_t zph = 0;    // bit b: parity of the next release of buffer b
            uint32_t zused = 0;  // bit b: buffer b was used before
            bool ok = true;
            for (int jc = jc0; jc < jc1 && ok; ++jc) {
                const int ck = chunk_len(jc);
                if (!wait_w(bfull, (uint32_t)((jc - jc0) & 1))) {
                    ok = false;
                    break;
                }
                for (int64_t pi = pre_lo; pi < pre_hi && ok; pi = unit_next(pi)) {
                    uint32_t bw = b_w0;
                    for (int q = 0; q < ck; ++q, bw += kBStep) {
                        const int qq = q % kChunkSteps;
                        const bool first = qq == 0;
                        const bool last = qq == kChunkSteps - 1 || q == ck - 1;
                        if (first && ((zused >> zb) & 1u)) {
                            // the epilogue has read this TMEM buffer's previous contents
                            if (!wait_w(&zempty[zb], (zph >> zb) & 1u)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                        }
                        // the producers arrive only after the stage's TMA copy landed
                        if (!wait_w(&op_full[slot], phase)) {
                            ok = false;
                            break;
                        }
                        const uint32_t dz = tmem + (uint32_t)(zb * BN);
#pragma unroll
                        for (int kk = 0; kk < 2; ++kk) {
                            const uint32_t adv = (uint32_t)kk * 2u;  // 8 tf32 = 32 bytes
                            mma_w(dz, ahi + adv, bw + adv, idesc, (first && kk == 0) ? 0u : 1u);
                            mma_w(dz, ahi + adv, bw + kBLo + adv, idesc, 1u);
                            mma_w(dz, alo + adv, bw + adv, idesc, 1u);
                        }
                        commit_w(&stage_empty[slot]);
                        if (last) {
                            if (a.withhold_signal && zused == 0 && zb == 0) {
                                // test hook: this buffer is never reported full, so the
                                // epilogue's bounded wait expires and the CTA aborts
                            } else {
                                commit_w(&zfull[zb]);
                            }
                            if ((zused >> zb) & 1u) zph ^= 1u << zb;
                            zused |= 1u << zb;
                            zb ^= 1;
                        }
                        if (++slot == NR) {
                            slot = 0;
                            phase ^= 1u;
                            ahi = a_hi0;
                            alo = a_lo0;
                        } else {
                            ahi += kAhiStep;
                            alo += kAloStep;
                        }
                    }
                }
                if (ok) commit_w(bempty);  // the B-chunk may be replaced once these finish
            }
            // all MMAs issued by this thread are complete before TMEM is freed
            commit_w(mma_done);
            if (lane == 0) wait_drain(mma_done, 0, a.status);
            if (kWarpIssue) __syncwarp();
        }
    } else if (warp < kFE) {
        // ---------------------- operand producers (64 threads) ----------------------
        const int ptid = tid - 64;   // 0 .. kPT - 1
        Ring<NR> rr;
        for (int64_t t = 0; t < T; ++t, rr.next()) {
            // the TMA refills a stage only after its MMAs finished, so the operand
            // tile of this stage is free once its raw tile has landed
            if (!warp_wait(&raw_full[rr.slot], rr.phase, abort_flag, a.status, kStatusTimeoutLo))
                break;
            const uint8_t* st = raw + rr.slot * L::kY;
            uint8_t* op = ops + rr.slot * L::kOp;
            if (!INNER) {
                // lo tile, elementwise at the same (swizzled) offsets as the raw tile
                const float4* src = reinterpret_cast<const float4*>(st);
                float4* dst = reinterpret_cast<float4*>(op);
                static_assert(INNER || (L::kY / 16) % kPT == 0, "whole rounds");
#pragma unroll
                for (int v = 0; v < (int)(L::kY / 16) / kPT; ++v) {
                    const int e = ptid + kPT * v;
                    const float4 x = src[e];
                    dst[e] = make_float4(tf32_lo(x.x), tf32_lo(x.y), tf32_lo(x.z), tf32_lo(x.w));
                }
            } else if (SMALL) {
                // staging tile is [ps][16 j][I i] (i contiguous): transpose into
                // K-major hi and lo rows slot * I + i; one 16-byte chunk (4 j) per
                // item, i fastest across lanes (consecutive loads, and the stores
                // of 8 consecutive rows hit 8 distinct bank groups)
                const float* stg = reinterpret_cast<const float*>(st);
                uint8_t* hi = op;
                uint8_t* lo = op + L::kA;
                const int Iv = (int)a.I;
                const int items = a.ps * Iv * 4;
                for (int u = ptid; u < items; u += kPT) {
                    const int i = u % Iv;
                    const int rest = u / Iv;
                    const int jc = rest & 3;
                    const int sl = rest >> 2;
                    const float* src = stg + (sl * kBK + 4 * jc) * Iv + i;
                    const float4 r = make_float4(src[0], src[Iv], src[2 * Iv], src[3 * Iv]);
                    const uint32_t off = sw64_off((uint32_t)(sl * Iv + i), (uint32_t)jc);
                    *reinterpret_cast<float4*>(hi + off) = r;
                    *reinterpret_cast<float4*>(lo + off) =
                        make_float4(tf32_lo(r.x), tf32_lo(r.y), tf32_lo(r.z), tf32_lo(r.w));
                }
            } else {
                // staging tile is [16 j][128 i] (i contiguous): transpose into the
                // K-major hi and lo tiles, one 4 (i) x 4 (j) block per thread and
                // round
                const float* stg = reinterpret_cast<const float*>(st);
                uint8_t* hi = op;
                uint8_t* lo = op + L::kA;
#pragma unroll
                for (int v = 0; v < (128 + kPT - 1) / kPT; ++v) {
                    const int blk = ptid + kPT * v;   // 128 blocks: 32 i-blocks x 4 j-chunks
                    if (128 % kPT != 0 && blk >= 128) break;
                    const int jc = blk & 3;
                    const int ib = blk >> 2;
                    float4 col[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        col[q] = *reinterpret_cast<const float4*>(stg + (4 * jc + q) * kBM + 4 * ib);
                    const float4 rows[4] = {make_float4(col[0].x, col[1].x, col[2].x, col[3].x),
                                            make_float4(col[0].y, col[1].y, col[2].y, col[3].y),
                                            make_float4(col[0].z, col[1].z, col[2].z, col[3].z),
                                            make_float4(col[0].w, col[1].w, col[2].w, col[3].w)};
#pragma unroll
                    for (int p = 0; p < 4; ++p) {
                        // Row 4 ib + p is stored at tile row
                        // 4 ib + (p ^ (ib & 1)), so that the 8 lanes of a quarter-warp
                        // (two i-blocks of opposite parity) hit 8 distinct bank groups;
                        // the epilogue undoes the swap
                        const int prow = p ^ (ib & 1);
                        const uint32_t off = sw64_off(4 * ib + prow, jc);
                        *reinterpret_cast<float4*>(hi + off) = rows[p];
                        *reinterpret_cast<float4*>(lo + off) =
                            make_float4(tf32_lo(rows[p].x), tf32_lo(rows[p].y), tf32_lo(rows[p].z),
                                        tf32_lo(rows[p].w));
                    }
                }
            }
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) mbar_arrive(&op_full[rr.slot]);
        }
    } else {
        // ---------------------- epilogue (16 warps) ----------------------
        if constexpr (SMALL) {
            // Tile row (TMEM lane) slot * I + i holds pre index pi_u + slot of the
            // unit; each warp's lanes span at most kW slots.  G rows of the next
            // unit are copied (cp.async) while the current one is drained; at the
            // end the slots are summed through shared memory.
            constexpr int kCols = BN / 4;
            constexpr int kLd = kEpiLd < kCols ? kEpiLd : kCols;  // TMEM columns per wait
            constexpr int kW = 3;
            const int quad = warp & 3;
            const int part = (warp - kFE) >> 2;
            const int64_t c0 = r0 + part * kCols;
            const int Iv = (int)a.I;
            const int lg = 32 * quad + lane;
            const int slot = lg / Iv;
            const int s_lo = (32 * quad) / Iv;
            float* gw = gsm + (warp - kFE) * 2 * kW * kCols;
            float acc[kCols];
#pragma unroll
            for (int e = 0; e < kCols; ++e) acc[e] = 0.f;
            auto fetch_g = [&](int64_t pu, int buf) {
                const int64_t pe = unit_next(pu);
                for (int e = lane; e < kW * kCols; e += 32) {
                    const int w = e / kCols, c = e - w * kCols;
                    const int64_t pi = pu + s_lo + w;
                    const bool in = (pi < pe) && (s_lo + w < a.ps) && (c0 + c < a.R);
                    const float* src = in ? a.gtab + pi * a.R + c0 + c : a.gtab;
                    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(
                                     smem_u32(gw + buf * kW * kCols + e)),
                                 "l"(src), "r"(in ? 4 : 0)
                                 : "memory");
                }
                asm volatile("cp.async.commit_group;" ::: "memory");
            };
            fetch_g(pre_lo, 0);
            int gb = 0;
            int zb = 0;
            uint32_t zph = 0;
            bool ok = true;
            for (int jc = jc0; jc < jc1 && ok; ++jc) {
                const int ck = chunk_len(jc);
                for (int64_t pi = pre_lo; pi < pre_hi && ok; pi = unit_next(pi)) {
                    asm volatile("cp.async.wait_group 0;" ::: "memory");
                    __syncwarp();
                    const int64_t pn = unit_next(pi);
                    fetch_g(pn < pre_hi ? pn : pre_lo, gb ^ 1);
                    const int srow = slot - s_lo < kW ? slot - s_lo : kW - 1;
                    const float* g_cur = gw + gb * kW * kCols + srow * kCols;
                    for (int q0 = 0; q0 < ck; q0 += kChunkSteps) {
                        if (!warp_wait(&zfull[zb], (zph >> zb) & 1u, abort_flag, a.status,
                                       kStatusTimeoutEpi)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t tbase =
                            tmem + ((uint32_t)(32 * quad) << 16) + (uint32_t)(zb * BN + part * kCols);
#pragma unroll
                        for (int cc = 0; cc < kCols; cc += kLd) {
                            uint32_t z[kLd];
                            tmem_ld_cols<kLd>(tbase + cc, z);
                            tmem_ld_wait();
#pragma unroll
                            for (int q = 0; q < kLd; ++q)
                                acc[cc + q] = fmaf(g_cur[cc + q], __uint_as_float(z[q]), acc[cc + q]);
                        }
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&zempty[zb]);
                        zph ^= 1u << zb;
                        zb ^= 1;
                    }
                    gb ^= 1;
                }
            }
            asm volatile("cp.async.wait_group 0;" ::: "memory");
            // sum the slots: rows slot * I + i of a [128][BN + 4] buffer over the
            // (now idle) B-chunk and stage area
            constexpr int kSP = BN + 4;
            float* S = reinterpret_cast<float*>(smem);
            const bool live = !*abort_flag;
            if (live) {
#pragma unroll
                for (int e = 0; e < kCols; e += 4)
                    *reinterpret_cast<float4*>(S + lg * kSP + part * kCols + e) =
                        make_float4(acc[e], acc[e + 1], acc[e + 2], acc[e + 3]);
            }
            asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * 32) : "memory");
            if (live) {
                float* dst = a.dst + (int64_t)blockIdx.z * a.dst_split_stride;
                for (int idx = tid - 32 * kFE; idx < Iv * BN; idx += kEpiWarps * 32) {
                    const int i = idx / BN, c = idx - i * BN;
                    if (r0 + c >= a.R) continue;
                    float sum = 0.f;
                    for (int sl = 0; sl < a.ps; ++sl) sum += S[(sl * Iv + i) * kSP + c];
                    dst[(int64_t)i * a.R + r0 + c] = sum;
                }
            }
        } else {
            // warp w reads TMEM lanes 32 * (w % 4) .. + 31 (rows) and a quarter of
            // the tile's columns.  The G(pi, :) row of the next (chunk, pi) pair is
            // copied into the warp's second G buffer (cp.async, no registers) while
            // the current pair is drained.
            constexpr int kCols = BN / 4;
            constexpr int kLd = kEpiLd < kCols ? kEpiLd : kCols;  // TMEM columns per wait
            const int quad = warp & 3;
            const int part = (warp - kFE) >> 2;
            const int lr = 32 * quad + lane;   // TMEM lane = tile row
            const int64_t row = m0 + (INNER ? (lr ^ ((lr >> 2) & 1)) : lr);
            const int64_t c0 = r0 + part * kCols;
            float* gw = gsm + (warp - kFE) * 2 * kCols;   // this warp's two G rows
            float acc[kCols];
#pragma unroll
            for (int e = 0; e < kCols; ++e) acc[e] = 0.f;
            auto fetch_g = [&](int64_t pi, int buf) {
                for (int e = lane; e < kCols; e += 32) {
                    const bool in = (c0 + e < a.R) && (pi < pre_hi);
                    const float* src = in ? a.gtab + pi * a.R + c0 + e : a.gtab;
                    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(
                                     smem_u32(gw + buf * kCols + e)),
                                 "l"(src), "r"(in ? 4 : 0)
                                 : "memory");
                }
                asm volatile("cp.async.commit_group;" ::: "memory");
            };
            fetch_g(pre_lo, 0);
            int gb = 0;           // G buffer of the current pair
            int zb = 0;           // TMEM buffer of the next unit
            uint32_t zph = 0;     // bit b: parity of the next completion of zfull[b]
            bool ok = true;
            for (int jc = jc0; jc < jc1 && ok; ++jc) {
                const int ck = chunk_len(jc);
                for (int64_t pi = pre_lo; pi < pre_hi && ok; ++pi) {
                    asm volatile("cp.async.wait_group 0;" ::: "memory");
                    __syncwarp();
                    fetch_g(pi + 1 < pre_hi ? pi + 1 : pre_lo, gb ^ 1);
                    const float* g_cur = gw + gb * kCols;
                    for (int q0 = 0; q0 < ck; q0 += kChunkSteps) {
                        if (!warp_wait(&zfull[zb], (zph >> zb) & 1u, abort_flag, a.status,
                                       kStatusTimeoutEpi)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t tbase =
                            tmem + ((uint32_t)(32 * quad) << 16) + (uint32_t)(zb * BN + part * kCols);
#pragma unroll
                        for (int cc = 0; cc < kCols; cc += kLd) {
                            uint32_t z[kLd];
                            tmem_ld_cols<kLd>(tbase + cc, z);
                            tmem_ld_wait();
#pragma unroll
                            for (int q = 0; q < kLd / 4; ++q) {
                                const float4 g = *reinterpret_cast<const float4*>(g_cur + cc + 4 * q);
                                acc[cc + 4 * q + 0] = fmaf(g.x, __uint_as_float(z[4 * q + 0]), acc[cc + 4 * q + 0]);
                                acc[cc + 4 * q + 1] = fmaf(g.y, __uint_as_float(z[4 * q + 1]), acc[cc + 4 * q + 1]);
                                acc[cc + 4 * q + 2] = fmaf(g.z, __uint_as_float(z[4 * q + 2]), acc[cc + 4 * q + 2]);
                                acc[cc + 4 * q + 3] = fmaf(g.w, __uint_as_float(z[4 * q + 3]), acc[cc + 4 * q + 3]);
                            }
                        }
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&zempty[zb]);
                        zph ^= 1u << zb;
                        zb ^= 1;
                    }
                    gb ^= 1;
                }
            }
            asm volatile("cp.async.wait_group 0;" ::: "memory");
            if (!*abort_flag && row < a.I) {
                float* dst = a.dst + (int64_t)blockIdx.z * a.dst_split_stride + row * a.R + c0;
                const bool vst = (a.R % 4 == 0) && ((reinterpret_cast<uintptr_t>(a.dst) & 15) == 0);
#pragma unroll
                for (int e = 0; e < kCols; e += 4) {
                    if (vst && c0 + e + 4 <= a.R) {
                        *reinterpret_cast<float4*>(dst + e) =
                            make_float4(acc[e], acc[e + 1], acc[e + 2], acc[e + 3]);
                    } else {
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            if (c0 + e + q < a.R) dst[e + q] = acc[e + q];
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols));
    }
}

// ---------------------------------------------------------------------------
// Tensor-core kernel with the A operand in tensor memory (large R)
// ---------------------------------------------------------------------------
// Four producer warps (one per TMEM lane quadrant) read their 32 rows of each
// raw Y tile from shared memory, one row per lane, split every value into tf32
// hi and lo and store both into tensor memory with tcgen05.st (lane = tile row,
// column = k).  The MMAs then read only B from shared memory: at full rate the
// tensor core otherwise takes most of the shared-memory bandwidth and starves
// the producers.  The innermost mode's i-contiguous tile needs no separate
// transpose (lane = row).  The raw tile is free as soon as the producers have
// read it, so the TMA ring is decoupled from the MMAs and runs far ahead.
// TMEM: accumulators at columns [0, BN) and [BN, 2 BN); A slots of 32 columns
// (hi 16 | lo 16) from column 2 BN.
constexpr int kTBN = 224;
constexpr int kTASlots = 2;
constexpr uint32_t kTACol0 = 2 * kTBN;
constexpr int kTProdWarps = 4;
constexpr int kTFirstEpi = 2 + kTProdWarps;
constexpr int kTThreads = (kTFirstEpi + kEpiWarps) * 32;

struct SmemT {
    static constexpr uint32_t kY = kBM * kBK * 4;      // 8 KB raw Y tile
    static constexpr uint32_t kB = kTBN * kBK * 4;     // 14 KB: one K-step of B (hi or lo)
    static constexpr int kCK = 4;                      // K-steps per B-chunk
    static constexpr uint32_t kBRes = kCK * 2 * kB;    // 112 KB resident B-chunk
    static constexpr int kRaw = 12;
    static constexpr uint32_t kG = kEpiWarps * 2 * (kTBN / 4) * 4;
    static constexpr uint32_t kBarBytes = 512;
    static constexpr uint32_t kOffRaw = kBRes;
    static constexpr uint32_t kOffG = kOffRaw + kRaw * kY;
    static constexpr uint32_t kOffBars = kOffG + kG;
    static constexpr uint32_t kTotal = 1024 + kOffBars + kBarBytes;
    static_assert(kTotal <= 232448, "shared memory budget");
    static_assert(kB % 512 == 0, "B tiles start on a swizzle-atom boundary");
    static_assert((2 * kRaw + 2 * kTASlots + 7) * 8 + 8 <= kBarBytes, "barrier area");
    static_assert(2 * kTBN + 32 * kTASlots <= 512, "TMEM columns");
};

template <bool INNER>
__global__ void __launch_bounds__(kTThreads, 1) tc_tmem_kernel(const __grid_constant__ TcArgs a) {
    using L = SmemT;
    constexpr int BN = kTBN;
    constexpr int CK = L::kCK;
    constexpr int NR = L::kRaw;
    constexpr int NA = kTASlots;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~(uintptr_t)1023);
    uint8_t* bres = smem;
    uint8_t* raw = smem + L::kOffRaw;
    float* gsm = reinterpret_cast<float*>(smem + L::kOffG);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kOffBars);
    uint64_t* raw_full = bars;                  // [NR] TMA landed
    uint64_t* raw_empty = raw_full + NR;        // [NR] producers read the tile
    uint64_t* a_full = raw_empty + NR;          // [NA] producers wrote the A slot
    uint64_t* a_empty = a_full + NA;            // [NA] MMAs that read the A slot are done
    uint64_t* zfull = a_empty + NA;             // [2]
    uint64_t* zempty = zfull + 2;               // [2]
    uint64_t* bfull = zempty + 2;               // [1]
    uint64_t* bempty = bfull + 1;               // [1]
    uint64_t* mma_done = bempty + 1;            // [1]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int64_t m0 = (int64_t)blockIdx.y * kBM;
    const int64_t r0 = (int64_t)blockIdx.x * BN;
    const int64_t pre_lo = (int64_t)blockIdx.z * a.pre_per_split;
    int64_t pre_hi = pre_lo + a.pre_per_split;
    if (pre_hi > a.npre) pre_hi = a.npre;
    const int64_t npi = pre_hi > pre_lo ? pre_hi - pre_lo : 0;
    const int KS = a.KS;
    const int njc = (KS + CK - 1) / CK;
    auto chunk_len = [&](int jc) { return min(CK, KS - jc * CK); };
    constexpr uint32_t kTmemCols = 512;

    if (tid == 0) {
        for (int s = 0; s < NR; ++s) {
            mbar_init(&raw_full[s], 1);
            mbar_init(&raw_empty[s], kTProdWarps);
        }
        for (int s = 0; s < NA; ++s) {
            mbar_init(&a_full[s], kTProdWarps);
            mbar_init(&a_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&zfull[b], 1);
            mbar_init(&zempty[b], kEpiWarps);
        }
        mbar_init(bfull, 1);
        mbar_init(bempty, 1);
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int64_t T = npi * KS;  // K-steps of this CTA

    if (warp == 0) {
        // ------------------------- TMA producer -------------------------
        if (lane == 0) {
            const uint8_t* bimg = reinterpret_cast<const uint8_t*>(a.bimg);
            Ring<NR> rr;
            int64_t issued = 0;
            int jc_loaded = -1;
            bool ok = true;
            auto load_b = [&](int jc) -> bool {
                if (jc > 0 && !wait_bounded(bempty, (uint32_t)((jc - 1) & 1), abort_flag, a.status,
                                            kStatusTimeoutTma))
                    return false;
                const int ck = chunk_len(jc);
                mbar_arrive_expect_tx(bfull, (uint32_t)(ck * 2 * L::kB));
                for (int q = 0; q < ck; ++q) {
                    const int ks = jc * CK + q;
                    const uint8_t* src = bimg + ((int64_t)blockIdx.x * KS + ks) * (int64_t)(2 * L::kB);
                    bulk_load(bres + q * 2 * L::kB, src, 2 * L::kB, bfull);
                }
                jc_loaded = jc;
                return true;
            };
            for (int jc = 0; jc < njc && ok; ++jc) {
                const int ck = chunk_len(jc);
                // the first NR Y tiles of chunk jc need only work of chunk jc - 1,
                // so they are issued before the chunk swap
                const int64_t swap_at = issued + NR;
                bool b_pending = true;
                for (int64_t pi = pre_lo; pi < pre_hi && ok; ++pi) {
                    const int cP = (int)(pi / a.nQ);
                    const int cQ = (int)(pi - (int64_t)cP * a.nQ);
                    for (int q = 0; q < ck; ++q, ++issued, rr.next()) {
                        if (b_pending && issued == swap_at) {
                            b_pending = false;
                            if (!load_b(jc)) {
                                ok = false;
                                break;
                            }
                        }
                        if (rr.reused && !wait_bounded(&raw_empty[rr.slot], rr.phase ^ 1u, abort_flag,
                                                       a.status, kStatusTimeoutTma)) {
                            ok = false;
                            break;
                        }
                        const int ks = jc * CK + q;
                        int role[kRoles];
                        if (INNER) {
                            role[kRoleJq] = ks * kBK;
                            role[kRoleJp] = 0;
                        } else {
                            const int jp = ks / a.jq_steps;
                            role[kRoleJq] = (ks - jp * a.jq_steps) * kBK;
                            role[kRoleJp] = jp;
                        }
                        role[kRoleI] = (int)m0;
                        role[kRolePP] = cP;
                        role[kRolePQ] = cQ;
                        int c[5];
                        tma_coords(a.slot, role, c);
                        mbar_arrive_expect_tx(&raw_full[rr.slot], a.y_box_bytes);
                        tma_load(&a.ymap, a.rank, c, raw + rr.slot * L::kY, &raw_full[rr.slot]);
                    }
                }
                if (ok && b_pending && !load_b(jc)) ok = false;
            }
            for (int64_t u = issued - 1; u >= 0 && u >= issued - NR; --u)
                wait_drain(&raw_full[u % NR], (uint32_t)((u / NR) & 1), a.status);
            if (jc_loaded >= 0) wait_drain(bfull, (uint32_t)(jc_loaded & 1), a.status);
        }
    } else if (warp == 1) {
        // ------------------------- MMA issuer -------------------------
        if (lane == 0) {
            const uint32_t idesc = (1u << 4) | (2u << 7) | (2u << 10) |
                                   ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);
            const uint32_t b_w0 = sdesc_lo(smem_u32(bres));
            constexpr uint32_t kBStep = (2 * L::kB) >> 4;
            constexpr uint32_t kBLo = L::kB >> 4;
            int as = 0;
            uint32_t aph = 0;
            int zb = 0;
            uint32_t zph = 0;
            uint32_t zused = 0;
            bool ok = true;
            for (int jc = 0; jc < njc && ok; ++jc) {
                const int ck = chunk_len(jc);
                if (!wait_bounded(bfull, (uint32_t)(jc & 1), abort_flag, a.status, kStatusTimeoutMma)) {
                    ok = false;
                    break;
                }
                for (int64_t pi = pre_lo; pi < pre_hi && ok; ++pi) {
                    uint32_t bw = b_w0;
                    for (int q = 0; q < ck; ++q, bw += kBStep) {
                        const int qq = q % kChunkSteps;
                        const bool first = qq == 0;
                        const bool last = qq == kChunkSteps - 1 || q == ck - 1;
                        if (first && ((zused >> zb) & 1u)) {
                            if (!wait_bounded(&zempty[zb], (zph >> zb) & 1u, abort_flag, a.status,
                                              kStatusTimeoutMma)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                        }
                        if (!wait_bounded(&a_full[as], aph, abort_flag, a.status, kStatusTimeoutMma)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t ta = tmem + kTACol0 + 32u * (uint32_t)as;
                        const uint32_t dz = tmem + (uint32_t)(zb * BN);
#pragma unroll
                        for (int kk = 0; kk < 2; ++kk) {
                            const uint32_t adv = (uint32_t)kk * 2u;   // 8 tf32 = 32 bytes of B
                            const uint32_t ac = (uint32_t)kk * 8u;    // 8 TMEM columns of A
                            mma_tf32_ta(dz, ta + ac, bw + adv, idesc, (first && kk == 0) ? 0u : 1u);
                            mma_tf32_ta(dz, ta + ac, bw + kBLo + adv, idesc, 1u);
                            mma_tf32_ta(dz, ta + 16u + ac, bw + adv, idesc, 1u);
                        }
                        mma_commit(&a_empty[as]);
                        if (last) {
                            if (a.withhold_signal && zused == 0 && zb == 0) {
                                // test hook: this buffer is never reported full
                            } else {
                                mma_commit(&zfull[zb]);
                            }
                            if ((zused >> zb) & 1u) zph ^= 1u << zb;
                            zused |= 1u << zb;
                            zb ^= 1;
                        }
                        if (++as == NA) {
                            as = 0;
                            aph ^= 1u;
                        }
                    }
                }
                if (ok) mma_commit(bempty);
            }
            mma_commit(mma_done);
            wait_drain(mma_done, 0, a.status);
        }
    } else if (warp < kTFirstEpi) {
        // --------------- operand producers: one TMEM lane quadrant each ---------------
        const int quad = warp & 3;
        const int r = 32 * quad + lane;   // tile row of this thread
        Ring<NR> rr;
        for (int64_t t = 0; t < T; ++t, rr.next()) {
            if (!warp_wait(&raw_full[rr.slot], rr.phase, abort_flag, a.status, kStatusTimeoutLo)) break;
            const uint8_t* st = raw + rr.slot * L::kY;
            uint32_t hi[16], lo[16];
            if (!INNER) {
                // row r of the K-major tile: 64 bytes, 64-byte swizzled
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const float4 v = *reinterpret_cast<const float4*>(st + sw64_off((uint32_t)r, (uint32_t)c));
                    hi[4 * c + 0] = __float_as_uint(v.x);
                    hi[4 * c + 1] = __float_as_uint(v.y);
                    hi[4 * c + 2] = __float_as_uint(v.z);
                    hi[4 * c + 3] = __float_as_uint(v.w);
                }
            } else {
                // column r of the [16 j][128 i] staging tile
                const float* stg = reinterpret_cast<const float*>(st);
#pragma unroll
                for (int j = 0; j < kBK; ++j) hi[j] = __float_as_uint(stg[j * kBM + r]);
            }
#pragma unroll
            for (int e = 0; e < kBK; ++e) lo[e] = __float_as_uint(tf32_lo(__uint_as_float(hi[e])));
            __syncwarp();
            if (lane == 0) mbar_arrive(&raw_empty[rr.slot]);   // the tile's values are in registers
            // A slot t % NA was last read by the MMAs of K-step t - NA
            const int as = (int)(t % NA);
            if (t >= NA && !warp_wait(&a_empty[as], (uint32_t)(((t / NA) - 1) & 1), abort_flag, a.status,
                                      kStatusTimeoutLo))
                break;
            tc_fence_after();
            const uint32_t ta = tmem + ((uint32_t)(32 * quad) << 16) + kTACol0 + 32u * (uint32_t)as;
            tmem_st16(ta, hi);
            tmem_st16(ta + 16u, lo);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&a_full[as]);
        }
    } else {
        // ---------------------- epilogue (16 warps) ----------------------
        constexpr int kCols = BN / 4;
        const int quad = warp & 3;
        const int part = (warp - kTFirstEpi) >> 2;
        const int64_t row = m0 + 32 * quad + lane;
        const int64_t c0 = r0 + part * kCols;
        float* gw = gsm + (warp - kTFirstEpi) * 2 * kCols;
        float acc[kCols];
#pragma unroll
        for (int e = 0; e < kCols; ++e) acc[e] = 0.f;
        auto fetch_g = [&](int64_t pi, int buf) {
            for (int e = lane; e < kCols; e += 32) {
                const bool in = (c0 + e < a.R) && (pi < pre_hi);
                const float* src = in ? a.gtab + pi * a.R + c0 + e : a.gtab;
                asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(
                                 smem_u32(gw + buf * kCols + e)),
                             "l"(src), "r"(in ? 4 : 0)
                             : "memory");
            }
            asm volatile("cp.async.commit_group;" ::: "memory");
        };
        fetch_g(pre_lo, 0);
        int gb = 0;
        int zb = 0;
        uint32_t zph = 0;
        bool ok = true;
        for (int jc = 0; jc < njc && ok; ++jc) {
            const int ck = chunk_len(jc);
            for (int64_t pi = pre_lo; pi < pre_hi && ok; ++pi) {
                asm volatile("cp.async.wait_group 0;" ::: "memory");
                __syncwarp();
                fetch_g(pi + 1 < pre_hi ? pi + 1 : pre_lo, gb ^ 1);
                const float* g_cur = gw + gb * kCols;
                for (int q0 = 0; q0 < ck; q0 += kChunkSteps) {
                    if (!warp_wait(&zfull[zb], (zph >> zb) & 1u, abort_flag, a.status, kStatusTimeoutEpi)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t tbase =
                        tmem + ((uint32_t)(32 * quad) << 16) + (uint32_t)(zb * BN + part * kCols);
#pragma unroll
                    for (int cc = 0; cc < kCols; cc += 8) {
                        uint32_t z[8];
                        tmem_ld8(tbase + cc, z);
                        tmem_ld_wait();
#pragma unroll
                        for (int q = 0; q < 2; ++q) {
                            const float4 g = *reinterpret_cast<const float4*>(g_cur + cc + 4 * q);
                            acc[cc + 4 * q + 0] = fmaf(g.x, __uint_as_float(z[4 * q + 0]), acc[cc + 4 * q + 0]);
                            acc[cc + 4 * q + 1] = fmaf(g.y, __uint_as_float(z[4 * q + 1]), acc[cc + 4 * q + 1]);
                            acc[cc + 4 * q + 2] = fmaf(g.z, __uint_as_float(z[4 * q + 2]), acc[cc + 4 * q + 2]);
                            acc[cc + 4 * q + 3] = fmaf(g.w, __uint_as_float(z[4 * q + 3]), acc[cc + 4 * q + 3]);
                        }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&zempty[zb]);
                    zph ^= 1u << zb;
                    zb ^= 1;
                }
                gb ^= 1;
            }
        }
        asm volatile("cp.async.wait_group 0;" ::: "memory");
        if (!*abort_flag && row < a.I) {
            float* dst = a.dst + (int64_t)blockIdx.z * a.dst_split_stride + row * a.R + c0;
            const bool vst = (a.R % 4 == 0) && ((reinterpret_cast<uintptr_t>(a.dst) & 15) == 0);
#pragma unroll
            for (int e = 0; e < kCols; e += 4) {
                if (vst && c0 + e + 4 <= a.R) {
                    *reinterpret_cast<float4*>(dst + e) = make_float4(acc[e], acc[e + 1], acc[e + 2], acc[e + 3]);
                } else {
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        if (c0 + e + q < a.R) dst[e + q] = acc[e + q];
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
    }
}

// ---------------------------------------------------------------------------
// Tensor-core kernel, two-term fp16 split (A in tensor memory, large R)
// ---------------------------------------------------------------------------
// Each fp32 value x (Y scaled by a power of two so that max|Y| < 2^14, and each
// Binner column likewise) is split into hi = fp16(x) and lo = fp16(x - hi); the
// three products hi*hi + hi*lo + lo*hi (kind::f16, fp32 accumulation) carry
// 2 x 11 significant bits, as the tf32 split does, with one K = 16 instruction
// per product per 16 contraction indices instead of two K = 8 ones.  The
// single MMA-issuing thread, which bounds the tf32 kernels, issues half as
// many instructions for the same work.  Structure as the tensor-memory-A tf32
// kernel; K-steps of 32 (128-byte rows of the raw fp32 tile, 64-byte rows of
// the fp16 B images).
constexpr int kBK2 = 32;
constexpr int kChunkSteps2 = 4;   // 128 contraction indices between TMEM drains

// Tile 128 x kH2BN; TMEM: accumulators at [0, BN) and [BN, 2 BN), then kH2Slots
// A slots of 32 columns (hi 16 | lo 16, one K-step each).  Producers and MMAs
// hand the slots over in groups of kH2Group K-steps (one barrier round trip per
// group), kH2Slots / kH2Group groups in flight.  Measured on 512^3, R = 2000:
// 128 x 224 with single-step groups (two slots) is the fastest per output
// column; 128 x 192 with four slots, in groups of one or two K-steps, was 9-11 %
// slower per column (the MMA issuer's per-step cost does not shrink with N).
// Warp roles.  The CTA is six warpgroups:
// producers (warps 0-3, one per TMEM lane quadrant), control (TMA warp 4, MMA
// warp 5, two idle warps), and four epilogue warpgroups (warps 8-23).  The
// control and producer warpgroups give registers back (setmaxnreg.dec) and the
// epilogue warpgroups take them (setmaxnreg.inc), so that the epilogue's
// register-resident accumulators do not spill.  The launch allots 80 registers
// a thread (768 threads); the split uses 128 x (56 + 72 + 4 x 88) = 61440 of
// the 61440 allotted, and the host refuses the launch if the kernel was built
// with fewer than 80.
constexpr int kH2ProdWarp0 = 0, kH2TmaWarp = 4, kH2MmaWarp = 5, kH2FirstEpi = 8;
constexpr int kH2Threads = (kH2FirstEpi + kEpiWarps) * 32;
constexpr int kH2RegsCtl = 56, kH2RegsProd = 72, kH2RegsEpi = 88;
constexpr int kH2RegsLaunch = 80;   // registers a thread the split needs at launch
static_assert(128 * (kH2RegsCtl + kH2RegsProd + 4 * kH2RegsEpi) <= kH2Threads * kH2RegsLaunch,
              "register split exceeds the launch allotment");
static_assert(kH2Threads == 768, "six warpgroups");

template <int N>
__device__ __forceinline__ void h2_regs_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void h2_regs_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
constexpr int kH2BN = 224;
constexpr int kH2Slots = (512 - 2 * kH2BN) / 32 < 4 ? (512 - 2 * kH2BN) / 32 : 4;
constexpr int kH2Group = 1;
constexpr uint32_t kH2ACol0 = 2 * kH2BN;
static_assert(kH2Slots >= 2 * kH2Group, "two A-slot groups in flight");

struct SmemH2 {
    static constexpr uint32_t kY = kBM * kBK2 * 4;     // 16 KB raw fp32 Y tile
    static constexpr uint32_t kB = kH2BN * kBK2 * 2;   // one K-step of B (hi or lo, fp16): BN x 64 B
    static constexpr int kCK = 4;                      // K-steps per B-chunk
    static constexpr uint32_t kBRes = kCK * 2 * kB;    // 112 KB resident B-chunk
    static constexpr int kRaw = 6;
    static constexpr uint32_t kG = kEpiWarps * 2 * (kH2BN / 4) * 4;
    static constexpr uint32_t kBarBytes = 512;
    static constexpr uint32_t kOffRaw = kBRes;
    static constexpr uint32_t kOffG = kOffRaw + kRaw * kY;
    static constexpr uint32_t kOffBars = kOffG + kG;
    static constexpr uint32_t kTotal = 1024 + kOffBars + kBarBytes;
    static_assert(kTotal <= 232448, "shared memory budget");
    static_assert(kB % 512 == 0 && kY % 1024 == 0, "swizzle-atom alignment");
    static_assert((2 * kRaw + 2 * 2 + 7) * 8 + 8 <= kBarBytes, "barrier area");
};

__device__ __forceinline__ uint32_t half2_bits(__half2 h) {
    uint32_t u;
    memcpy(&u, &h, sizeof(u));
    return u;
}

// Scale of the Y entries of pre index pi, or of output row `row` when the slab
// is the row; and the factor that undoes the scale of output row `row` at the
// end (the global scale unless the slab is the row: G absorbs the rest).
__device__ __forceinline__ float y_scale_pre(const TcArgs& a, int64_t pi) {
    return slab_scale(a.slab_bits, pi / a.slab_div, *a.ymax_bits);
}
__device__ __forceinline__ float y_scale_row(const TcArgs& a, int64_t row) {
    return slab_scale(a.slab_bits, row < a.I ? row : a.I - 1, *a.ymax_bits);
}
__device__ __forceinline__ float y_unscale(const TcArgs& a, int64_t row) {
    return pow2_recip(a.slab_rows ? y_scale_row(a, row) : pow2_scale(*a.ymax_bits));
}

// D (+)= A * B, kind::f16, A (M=128 rows = lanes, 8 columns = 16 fp16 of K) in
// tensor memory, B by descriptor low word (high word constant)
__device__ __forceinline__ void mma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t idesc,
                                           uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t.reg .b64 db;\n\t"
        "mov.b64 db, {%2, %3};\n\t"
        "setp.ne.b32 p, %5, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], db, %4, p;\n\t}\n" ::"r"(d_tmem),
        "r"(a_tmem), "r"(b_lo), "r"((uint32_t)(kDescSw64Hi >> 32)), "r"(idesc), "r"(acc));
}

template <bool INNER>
__global__ void __launch_bounds__(kH2Threads, 1) tc_h2_kernel(const __grid_constant__ TcArgs a) {
    using L = SmemH2;
    constexpr int BN = kH2BN;
    constexpr int CK = L::kCK;
    constexpr int NR = L::kRaw;
    constexpr int NG = kH2Slots / kH2Group;   // A-slot groups in flight
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~(uintptr_t)1023);
    uint8_t* bres = smem;
    uint8_t* raw = smem + L::kOffRaw;
    float* gsm = reinterpret_cast<float*>(smem + L::kOffG);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kOffBars);
    uint64_t* raw_full = bars;                  // [NR] TMA landed
    uint64_t* raw_empty = raw_full + NR;        // [NR] producers read the tile
    uint64_t* a_full = raw_empty + NR;          // [NG] producers wrote the group's A slots
    uint64_t* a_empty = a_full + NG;            // [NG] MMAs that read the group's A slots are done
    uint64_t* zfull = a_empty + NG;             // [2]
    uint64_t* zempty = zfull + 2;               // [2]
    uint64_t* bfull = zempty + 2;               // [1]
    uint64_t* bempty = bfull + 1;               // [1]
    uint64_t* mma_done = bempty + 1;            // [1]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int64_t m0 = (int64_t)blockIdx.y * kBM;
    const int64_t r0 = (int64_t)blockIdx.x * BN;
    const int64_t pre_lo = (int64_t)blockIdx.z * a.pre_per_split;
    int64_t pre_hi = pre_lo + a.pre_per_split;
    if (pre_hi > a.npre) pre_hi = a.npre;
    const int KS = a.KS;
    const int njc = (KS + CK - 1) / CK;
    auto chunk_len = [&](int jc) { return min(CK, KS - jc * CK); };
    constexpr uint32_t kTmemCols = 512;

    if (tid == 0) {
        for (int s = 0; s < NR; ++s) {
            mbar_init(&raw_full[s], 1);
            mbar_init(&raw_empty[s], kTProdWarps);
        }
        for (int s = 0; s < NG; ++s) {
            mbar_init(&a_full[s], kTProdWarps);
            mbar_init(&a_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&zfull[b], 1);
            mbar_init(&zempty[b], kEpiWarps);
        }
        mbar_init(bfull, 1);
        mbar_init(bempty, 1);
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kH2MmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const bool prod_warp = warp >= kH2ProdWarp0 && warp < kH2ProdWarp0 + kTProdWarps;
    if (!prod_warp && warp < kH2FirstEpi) {
        // control warpgroup: TMA warp, MMA warp and two idle warps
        h2_regs_dec<kH2RegsCtl>();
        if (warp == kH2TmaWarp) {
            // ------------------------- TMA producer -------------------------
            if (lane == 0) {
                const uint8_t* bimg = reinterpret_cast<const uint8_t*>(a.bimg);
                Ring<NR> rr;
                int64_t issued = 0;
                int jc_loaded = -1;
                bool ok = true;
                auto load_b = [&](int jc) -> bool {
                    if (jc > 0 && !wait_bounded_inl(bempty, (uint32_t)((jc - 1) & 1), abort_flag, a.status,
                                                kStatusTimeoutTma))
                        return false;
                    const int ck = chunk_len(jc);
                    mbar_arrive_expect_tx(bfull, (uint32_t)(ck * 2 * L::kB));
                    for (int q = 0; q < ck; ++q) {
                        const int ks = jc * CK + q;
                        const uint8_t* src = bimg + ((int64_t)blockIdx.x * KS + ks) * (int64_t)(2 * L::kB);
                        bulk_load(bres + q * 2 * L::kB, src, 2 * L::kB, bfull);
                    }
                    jc_loaded = jc;
                    return true;
                };
                for (int jc = 0; jc < njc && ok; ++jc) {
                    const int ck = chunk_len(jc);
                    // the first NR Y tiles of chunk jc need only work of chunk jc - 1,
                    // so they are issued before the chunk swap
                    const int64_t swap_at = issued + NR;
                    bool b_pending = true;
                    for (int64_t pi = pre_lo; pi < pre_hi && ok; ++pi) {
                        const int cP = (int)(pi / a.nQ);
                        const int cQ = (int)(pi - (int64_t)cP * a.nQ);
                        for (int q = 0; q < ck; ++q, ++issued, rr.next()) {
                            if (b_pending && issued == swap_at) {
                                b_pending = false;
                                if (!load_b(jc)) {
                                    ok = false;
                                    break;
                                }
                            }
                            if (rr.reused && !wait_bounded_inl(&raw_empty[rr.slot], rr.phase ^ 1u, abort_flag,
                                                           a.status, kStatusTimeoutTma)) {
                                ok = false;
                                break;
                            }
                            const int ks = jc * CK + q;
                            int role[kRoles];
                            if (INNER) {
                                role[kRoleJq] = ks * kBK2;
                                role[kRoleJp] = 0;
                            } else {
                                const int jp = ks / a.jq_steps;
                                role[kRoleJq] = (ks - jp * a.jq_steps) * kBK2;
                                role[kRoleJp] = jp;
                            }
                            role[kRoleI] = (int)m0;
                            role[kRolePP] = cP;
                            role[kRolePQ] = cQ;
                            int c[5];
                            tma_coords(a.slot, role, c);
                            mbar_arrive_expect_tx(&raw_full[rr.slot], a.y_box_bytes);
                            tma_load(&a.ymap, a.rank, c, raw + rr.slot * L::kY, &raw_full[rr.slot]);
                        }
                    }
                    if (ok && b_pending && !load_b(jc)) ok = false;
                }
                for (int64_t u = issued - 1; u >= 0 && u >= issued - NR; --u)
                    wait_drain_inl(&raw_full[u % NR], (uint32_t)((u / NR) & 1), a.status);
                if (jc_loaded >= 0) wait_drain_inl(bfull, (uint32_t)(jc_loaded & 1), a.status);
            }
        } else if (warp == kH2MmaWarp) {
            // ------------------------- MMA issuer -------------------------
            if (lane == 0) {
                // kind::f16: fp16 A and B, fp32 accumulator
                const uint32_t idesc = (1u << 4) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);
                const uint32_t b_w0 = sdesc_lo(smem_u32(bres));
                constexpr uint32_t kBStep = (2 * L::kB) >> 4;
                constexpr uint32_t kBLo = L::kB >> 4;
                int ag = 0;             // A-slot group of the current K-step (ring of NG)
                uint32_t aph = 0;
                bool a_ready = false;   // a_full[ag] already observed complete (prefetched test)
                int zb = 0;
                uint32_t zph = 0;
                uint32_t zused = 0;
                bool ok = true;
                for (int jc = 0; jc < njc && ok; ++jc) {
                    const int ck = chunk_len(jc);
                    if (!wait_bounded_inl(bfull, (uint32_t)(jc & 1), abort_flag, a.status, kStatusTimeoutMma)) {
                        ok = false;
                        break;
                    }
                    for (int64_t pi = pre_lo; pi < pre_hi && ok; ++pi) {
                        uint32_t bw = b_w0;
                        for (int q = 0; q < ck; ++q, bw += kBStep) {
                            const int qq = q % kChunkSteps2;
                            const bool first = qq == 0;
                            const bool last = qq == kChunkSteps2 - 1 || q == ck - 1;
                            if (first && ((zused >> zb) & 1u)) {
                                if (!wait_bounded_inl(&zempty[zb], (zph >> zb) & 1u, abort_flag, a.status,
                                                  kStatusTimeoutMma)) {
                                    ok = false;
                                    break;
                                }
                                tc_fence_after();
                            }
                            // a group is kH2Group consecutive K-steps of one unit
                            const bool gstart = q % kH2Group == 0;
                            const bool gend = q % kH2Group == kH2Group - 1 || q == ck - 1;
                            if (gstart) {
                                if (!a_ready && !wait_bounded_inl(&a_full[ag], aph, abort_flag, a.status, kStatusTimeoutMma)) {
                                    ok = false;
                                    break;
                                }
                                tc_fence_after();
                            }
                            const uint32_t ta =
                                tmem + kH2ACol0 + 32u * (uint32_t)(ag * kH2Group + q % kH2Group);
                            const uint32_t dz = tmem + (uint32_t)(zb * BN);
#pragma unroll
                            for (int kk = 0; kk < 2; ++kk) {
                                const uint32_t adv = (uint32_t)kk * 2u;   // 16 fp16 = 32 bytes of B
                                const uint32_t ac = (uint32_t)kk * 8u;    // 8 TMEM columns (16 fp16) of A
                                mma_f16_ta(dz, ta + ac, bw + adv, idesc, (first && kk == 0) ? 0u : 1u);
                                mma_f16_ta(dz, ta + ac, bw + kBLo + adv, idesc, 1u);
                                mma_f16_ta(dz, ta + 16u + ac, bw + adv, idesc, 1u);
                            }
                            if (gend) mma_commit(&a_empty[ag]);
                            if (last) {
                                if (a.withhold_signal && zused == 0 && zb == 0) {
                                    // test hook: this buffer is never reported full
                                } else {
                                    mma_commit(&zfull[zb]);
                                }
                                if ((zused >> zb) & 1u) zph ^= 1u << zb;
                                zused |= 1u << zb;
                                zb ^= 1;
                            }
                            if (gend) {
                                if (++ag == NG) {
                                    ag = 0;
                                    aph ^= 1u;
                                }
                                // non-blocking test of the next group; its answer is used at
                                // the next group start, so its latency overlaps the bookkeeping
                                a_ready = mbar_test_wait(&a_full[ag], aph) != 0;
                            }
                        }
                    }
                    if (ok) mma_commit(bempty);
                }
                mma_commit(mma_done);
                wait_drain_inl(mma_done, 0, a.status);
            }
        }
    } else if (prod_warp) {
        h2_regs_dec<kH2RegsProd>();
        // --------------- operand producers: one TMEM lane quadrant each ---------------
        const int quad = warp & 3;
        const int r = 32 * quad + lane;   // tile row of this thread
        // Y is scaled by a power of two: per row (mode 0 with per-slab scales) or
        // per pre index
        const float sy_row = a.slab_rows ? y_scale_row(a, m0 + r) : 1.f;
        float sy = sy_row;
        Ring<NR> rr;
        int ag = 0;          // A-slot group of the current K-step (ring of NG)
        int64_t g = 0;       // groups started so far
        bool ok = true;
        for (int jc = 0; jc < njc && ok; ++jc) {
            const int ck = chunk_len(jc);
            for (int64_t pi = pre_lo; pi < pre_hi && ok; ++pi) {
                if (!a.slab_rows) sy = y_scale_pre(a, pi);
                for (int q = 0; q < ck; ++q, rr.next()) {
                    const bool gstart = q % kH2Group == 0;
                    const bool gend = q % kH2Group == kH2Group - 1 || q == ck - 1;
                    if (!warp_wait_inl(&raw_full[rr.slot], rr.phase, abort_flag, a.status, kStatusTimeoutLo)) {
                        ok = false;
                        break;
                    }
                    if (gstart) {
                        // the group's slots were last read by the MMAs of group g - NG
                        if (g >= NG && !warp_wait_inl(&a_empty[ag], (uint32_t)(((g / NG) - 1) & 1), abort_flag,
                                                  a.status, kStatusTimeoutLo)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                    }
                    const uint8_t* st = raw + rr.slot * L::kY;
                    const uint32_t ta = tmem + ((uint32_t)(32 * quad) << 16) + kH2ACol0 +
                                        32u * (uint32_t)(ag * kH2Group + q % kH2Group);
                    // two halves of 16 contraction indices: hi to columns [8h, 8h + 8), lo
                    // to [16 + 8h, 16 + 8h + 8); column c holds k = 2c (low half), 2c + 1
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        float v[16];
                        if (!INNER) {
                            // row r of the K-major tile: 128 bytes, 128-byte swizzled
#pragma unroll
                            for (int c = 0; c < 4; ++c) {
                                const int cc = 4 * h + c;
                                const float4 x = *reinterpret_cast<const float4*>(
                                    st + (uint32_t)r * 128u + ((((uint32_t)cc ^ (uint32_t)r) & 7u) << 4));
                                v[4 * c + 0] = x.x;
                                v[4 * c + 1] = x.y;
                                v[4 * c + 2] = x.z;
                                v[4 * c + 3] = x.w;
                            }
                        } else {
                            // column r of the [32 j][128 i] staging tile
                            const float* stg = reinterpret_cast<const float*>(st);
#pragma unroll
                            for (int j = 0; j < 16; ++j) v[j] = stg[(16 * h + j) * kBM + r];
                        }
                        uint32_t hi[8], lo[8];
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            // packed conversions: hi = fp16x2(x), lo = fp16x2(x - hi)
                            // (x - hi is exact in fp32)
                            const float x0 = v[2 * c] * sy, x1 = v[2 * c + 1] * sy;
                            const __half2 hh = __floats2half2_rn(x0, x1);
                            const float2 hf = __half22float2(hh);
                            const __half2 ll = __floats2half2_rn(x0 - hf.x, x1 - hf.y);
                            hi[c] = half2_bits(hh);
                            lo[c] = half2_bits(ll);
                        }
                        tmem_st8(ta + 8u * (uint32_t)h, hi);
                        tmem_st8(ta + 16u + 8u * (uint32_t)h, lo);
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&raw_empty[rr.slot]);   // the tile has been read
                    if (gend) {
                        tmem_st_wait();
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&a_full[ag]);
                        ++g;
                        if (++ag == NG) ag = 0;
                    }
                }
            }
        }
    } else {
        h2_regs_inc<kH2RegsEpi>();
        // ---------------------- epilogue (16 warps) ----------------------
        constexpr int kCols = BN / 4;
        const int quad = warp & 3;
        const int part = (warp - kH2FirstEpi) >> 2;
        const int64_t row = m0 + 32 * quad + lane;
        const int64_t c0 = r0 + part * kCols;
        float* gw = gsm + (warp - kH2FirstEpi) * 2 * kCols;
        float acc[kCols];
#pragma unroll
        for (int e = 0; e < kCols; ++e) acc[e] = 0.f;
        auto fetch_g = [&](int64_t pi, int buf) {
            for (int e = lane; e < kCols; e += 32) {
                const bool in = (c0 + e < a.R) && (pi < pre_hi);
                const float* src = in ? a.gtab + pi * a.R + c0 + e : a.gtab;
                asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(
                                 smem_u32(gw + buf * kCols + e)),
                             "l"(src), "r"(in ? 4 : 0)
                             : "memory");
            }
            asm volatile("cp.async.commit_group;" ::: "memory");
        };
        fetch_g(pre_lo, 0);
        int gb = 0;
        int zb = 0;
        uint32_t zph = 0;
        bool ok = true;
        for (int jc = 0; jc < njc && ok; ++jc) {
            const int ck = chunk_len(jc);
            for (int64_t pi = pre_lo; pi < pre_hi && ok; ++pi) {
                asm volatile("cp.async.wait_group 0;" ::: "memory");
                __syncwarp();
                fetch_g(pi + 1 < pre_hi ? pi + 1 : pre_lo, gb ^ 1);
                const float* g_cur = gw + gb * kCols;
                for (int q0 = 0; q0 < ck; q0 += kChunkSteps) {
                    if (!warp_wait_inl(&zfull[zb], (zph >> zb) & 1u, abort_flag, a.status, kStatusTimeoutEpi)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t tbase =
                        tmem + ((uint32_t)(32 * quad) << 16) + (uint32_t)(zb * BN + part * kCols);
#pragma unroll
                    for (int cc = 0; cc < kCols; cc += kH2EpiLd) {
                        uint32_t z[kH2EpiLd];
                        if constexpr (kH2EpiLd == 8)
                            tmem_ld8(tbase + cc, z);
                        else
                            tmem_ld4(tbase + cc, z);
                        tmem_ld_wait();
#pragma unroll
                        for (int q = 0; q < kH2EpiLd / 4; ++q) {
                            const float4 g = *reinterpret_cast<const float4*>(g_cur + cc + 4 * q);
                            acc[cc + 4 * q + 0] = fmaf(g.x, __uint_as_float(z[4 * q + 0]), acc[cc + 4 * q + 0]);
                            acc[cc + 4 * q + 1] = fmaf(g.y, __uint_as_float(z[4 * q + 1]), acc[cc + 4 * q + 1]);
                            acc[cc + 4 * q + 2] = fmaf(g.z, __uint_as_float(z[4 * q + 2]), acc[cc + 4 * q + 2]);
                            acc[cc + 4 * q + 3] = fmaf(g.w, __uint_as_float(z[4 * q + 3]), acc[cc + 4 * q + 3]);
                        }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&zempty[zb]);
                    zph ^= 1u << zb;
                    zb ^= 1;
                }
                gb ^= 1;
            }
        }
        asm volatile("cp.async.wait_group 0;" ::: "memory");
        if (!*abort_flag && row < a.I && a.ttm_q > 0) {
            // mode-n product: column j of row (p, q) is T[p, j, q]; the lanes of a
            // warp hold consecutive q, so each store instruction writes 128 bytes
            const float inv_y = y_unscale(a, row);
            const int64_t p = row / a.ttm_q, q = row - p * a.ttm_q;
            float* dst = a.dst + p * a.R * a.ttm_q + q;
#pragma unroll
            for (int e = 0; e < kCols; ++e)
                if (c0 + e < a.R) dst[(c0 + e) * a.ttm_q] = acc[e] * inv_y * pow2_recip(a.colscale[c0 + e]);
        } else if (!*abort_flag && row < a.I) {
            // undo the power-of-two scales of Y and of each Binner column (exact)
            const float inv_y = y_unscale(a, row);
            float* dst = a.dst + (int64_t)blockIdx.z * a.dst_split_stride + row * a.R + c0;
            const bool vst = (a.R % 4 == 0) && ((reinterpret_cast<uintptr_t>(a.dst) & 15) == 0);
#pragma unroll
            for (int e = 0; e < kCols; e += 4) {
                float v[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float cs = (c0 + e + q < a.R) ? a.colscale[c0 + e + q] : 1.f;
                    v[q] = acc[e + q] * inv_y * pow2_recip(cs);
                }
                if (vst && c0 + e + 4 <= a.R) {
                    *reinterpret_cast<float4*>(dst + e) = make_float4(v[0], v[1], v[2], v[3]);
                } else {
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        if (c0 + e + q < a.R) dst[e + q] = v[q];
                }
                asm volatile("" ::: "memory");   // keep one group of column scales in flight
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kH2MmaWarp) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
    }
}


// ---------------------------------------------------------------------------
// Two-term fp16 split with both operands in shared memory.  Y is split once per
// call into fp16 hi and lo images laid out like Y (split_image_kernel); the
// kernel streams 128-row x 64-index tiles of both images with TMA (128-byte
// swizzle) and issues, per 16 contraction indices, hi*Bhi + hi*Blo + lo*Bhi into
// a TMEM accumulator.  Same arithmetic as tc_h2_kernel, but no producer warps:
// the only hand-over per K-step (64 indices, twelve MMAs) is TMA -> MMA.
// Roles: warp 0 TMA, warp 1 MMA, warps 2-3 idle (the control warpgroup, which
// gives registers back), warps 4-19 epilogue (which take them); the variant
// that converts Y in place adds converter warps 4-7 and moves the epilogue to
// warps 8-23.
// ---------------------------------------------------------------------------
constexpr int kBK4 = 64;          // contraction indices per K-step (128-byte fp16 rows)
constexpr int kImgCK = 2;   // K-steps per B chunk and per TMEM drain (128 indices)
constexpr int kImgEpiWarp0 = 4;
constexpr int kImgThreads = (kImgEpiWarp0 + kEpiWarps) * 32;   // 640
// registers a thread: the launch allots 96 (65536 / 640, in units of 8); the
// split uses 128 x (56 + 4 x 104) = 60416 of the 61440 allotted
constexpr int kImgRegsCtl = 56, kImgRegsEpi = 104, kImgRegsLaunch = 96;
static_assert(128 * (kImgRegsCtl + 4 * kImgRegsEpi) <= kImgThreads * kImgRegsLaunch, "register split");
// in-place conversion adds a warpgroup of four converter warps (warps 4-7; the
// epilogue moves to warps 8-23): 768 threads, 80 registers a thread at launch,
// split 56 (control) + 40 (converters) + 4 x 96 (epilogue), 61440 in all
constexpr int kCvtEpiWarp0 = 8;
constexpr int kCvtThreads = (kCvtEpiWarp0 + kEpiWarps) * 32;   // 768
constexpr int kCvtRegsCtl = 56, kCvtRegsCvt = 40, kCvtRegsEpi = 96, kCvtRegsLaunch = 80;
static_assert(128 * (kCvtRegsCtl + kCvtRegsCvt + 4 * kCvtRegsEpi) <= kCvtThreads * kCvtRegsLaunch,
              "register split");
static_assert(kCvtThreads * kCvtRegsLaunch <= 65536, "register file");

// K-major, 128-byte swizzle descriptor: 8-row groups of 128-byte rows, 1024
// bytes apart (high word; the low word is the start address >> 4 and LBO = 1)
constexpr uint64_t kDescSw128Hi = ((uint64_t)1 << 16)            // leading byte offset (unused)
                                | ((uint64_t)(1024 >> 4) << 32)  // stride byte offset: 8 rows x 128 B
                                | ((uint64_t)1 << 46)            // descriptor version
                                | ((uint64_t)2 << 61);           // 128-byte swizzle

__device__ __forceinline__ uint32_t sdesc128_lo(uint32_t saddr) {
    return (uint32_t)kDescSw128Hi | ((saddr & 0x3FFFFu) >> 4);
}

// D (+)= A * B, kind::f16, both operands by descriptor low word (128-byte swizzle)
__device__ __forceinline__ void mma_f16_ss(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo, uint32_t idesc,
                                           uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t.reg .b64 da, db;\n\t"
        "mov.b64 da, {%1, %3};\n\t"
        "mov.b64 db, {%2, %3};\n\t"
        "setp.ne.b32 p, %5, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %4, p;\n\t}\n" ::"r"(d_tmem),
        "r"(a_lo), "r"(b_lo), "r"((uint32_t)(kDescSw128Hi >> 32)), "r"(idesc), "r"(acc));
}

template <int N>
__device__ __forceinline__ void regs_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void regs_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

template <int BN, bool SMALL = false>
struct SmemImg {
    static constexpr uint32_t kA = kBM * 128;      // 16 KB: one image tile (128 rows x 64 fp16)
    static constexpr uint32_t kStage = 2 * kA;     // hi and lo tiles
    static constexpr uint32_t kB = BN * 128;       // one K-step of B (hi or lo)
    static constexpr uint32_t kBRes = kImgCK * 2 * kB;
    // barriers in the first 512 bytes, then (in-place conversion) the scales of
    // the row tile's 128 rows, then the reciprocals of the tile's column scales
    static constexpr uint32_t kBarBytes = 2048;
    static constexpr uint32_t kFree = 232448u - 1024u - kBarBytes - kBRes;
    static constexpr int kStages = kFree / kStage > 6 ? 6 : (int)(kFree / kStage);
    // small I: the slot sums at the end go through a [128][BN + 4] fp32 buffer
    // laid over the (then idle) B chunk and operand stages
    static_assert(!SMALL || (uint32_t)(kBM * (BN + 4) * 4) <= kBRes + kStages * kStage, "slot-sum buffer");
    static constexpr uint32_t kOffA = kBRes;
    static constexpr uint32_t kOffBars = kOffA + kStages * kStage;
    static constexpr uint32_t kTotal = 1024 + kOffBars + kBarBytes;
    static_assert(kStages >= 3, "operand ring depth");
    static_assert(kTotal <= 232448, "shared memory budget");
    static_assert(kB % 1024 == 0, "swizzle-atom alignment");
    static_assert((3 * kStages + 7) * 8 + 8 <= 512, "barrier area");
};

// MN-major A operand (the innermost mode from the natural images, MN = true):
// each image tile is two TMA boxes of 64 i (128 bytes, contiguous in the image)
// x 64 contraction indices, 8 KB apart, which is the canonical MN-major layout
// with a 128-byte swizzle: 8-row groups of K 1024 bytes apart (stride offset),
// the two 64-row halves of M 8192 bytes apart (leading offset); a slice of 16
// contraction indices advances the start address by 16 rows (2048 bytes).
constexpr uint32_t kDescMnLo = (uint32_t)((8192 >> 4) << 16);   // leading byte offset: M halves

__device__ __forceinline__ uint32_t sdesc128mn_lo(uint32_t saddr) { return kDescMnLo | ((saddr & 0x3FFFFu) >> 4); }

// CVT = true: the operand stages are filled from fp32 Y instead of the images
// (the first mode of a call, which then also writes the images).  The TMA warp
// loads each K-step as two 32-index fp32 boxes (128-byte swizzle) into the
// stage; warps 4-7 (32 rows each) convert it in place into the hi and lo
// tiles, with the same split and scales as split_image_kernel, and release it
// to the MMA warp; the TMA warp stores each converted tile to the images
// (column tile 0 only; other column tiles read the same Y) once it is
// converted, checking the tile it loaded NS - 1 loads earlier after each load,
// and waits for a store's reads before it refills that stage.  Every row's fp32 bytes and its hi and lo bytes lie in that row's
// 128-byte lines of the two halves of the stage, so one warp owns all the
// bytes of its rows and loads them before it stores.  A scaled value outside
// the fp16 range sets *a.ovf.
template <int BN, bool SMALL, bool MN, bool CVT = false>
__global__ void __launch_bounds__(CVT ? kCvtThreads : kImgThreads, 1) tc_img_kernel(const __grid_constant__ TcArgs a) {
    constexpr int EW0 = CVT ? kCvtEpiWarp0 : kImgEpiWarp0;   // first epilogue warp
    static_assert(!(SMALL && MN), "stacked tiles read K-major images");
    static_assert(!CVT || (!SMALL && !MN), "in-place conversion: natural K-major tiles");
    if (a.enable != nullptr && *a.enable == 0) return;
    using L = SmemImg<BN, SMALL>;
    constexpr int NS = L::kStages;
    constexpr int CK = kImgCK;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~(uintptr_t)1023);
    uint8_t* bres = smem;
    uint8_t* ring = smem + L::kOffA;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kOffBars);
    uint64_t* full = bars;                      // [NS] both image tiles of the stage landed
    uint64_t* empty = full + NS;                // [NS] the MMAs that read the stage are done
    uint64_t* zfull = empty + NS;               // [2]
    uint64_t* zempty = zfull + 2;               // [2]
    uint64_t* bfull = zempty + 2;               // [1]
    uint64_t* bempty = bfull + 1;               // [1]
    uint64_t* mma_done = bempty + 1;            // [1]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    uint64_t* yfull = mma_done + 2;             // [NS] (CVT) the fp32 boxes of the stage landed
    float* sscale = reinterpret_cast<float*>(smem + L::kOffBars + 512);   // [128] (CVT) row scales
    float* colinv = reinterpret_cast<float*>(smem + L::kOffBars + 1024);  // [BN] 1 / column scale
    static_assert(BN * 4 <= 1024, "column-scale area");

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int64_t r0 = (int64_t)blockIdx.x * BN;
    const int KS = a.KS;
    const int njc = (KS + CK - 1) / CK;
    const Share share = cta_share(a, njc);
    const int64_t pre_lo = share.pre_lo, pre_hi = share.pre_hi;
    const int jc0 = share.jc0, jc1 = share.jc1;
    auto chunk_len = [&](int jc) { return min(CK, KS - jc * CK); };
    // row tiles of this CTA: blockIdx.y alone, or (persistent) every gridDim.y-th
    // one; every role walks the same sequence, and the pipeline (operand ring,
    // accumulator buffers, B chunks) runs on across tiles
    const int64_t ty_end = (a.tiles_y > 0 && !SMALL) ? a.tiles_y : (int64_t)blockIdx.y + 1;
    const int64_t ty_step = (a.tiles_y > 0 && !SMALL) ? (int64_t)gridDim.y : 1;
    constexpr uint32_t kTmemCols = 2 * BN;   // two accumulator buffers
    static_assert(kTmemCols >= 32 && kTmemCols <= 512 && (kTmemCols & (kTmemCols - 1)) == 0,
                  "TMEM allocation: a power of two in [32, 512]");

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], CVT ? 4 : 1);   // CVT: the four converter warps
            mbar_init(&empty[s], 1);
            if (CVT) mbar_init(&yfull[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&zfull[b], 1);
            mbar_init(&zempty[b], kEpiWarps);
        }
        mbar_init(bfull, 1);
        mbar_init(bempty, 1);
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // Work units: one pre index, or (small I) up to ps consecutive pre indices
    // stacked in one 128-row tile (rows slot * I + i), never crossing a multiple
    // of batch_len.
    auto unit_next = [&](int64_t pi) -> int64_t {
        if (!SMALL) return pi + 1;
        int64_t e = pi + a.ps;
        const int64_t row_end = (pi / a.batch_len + 1) * a.batch_len;
        if (e > row_end) e = row_end;
        return e < pre_hi ? e : pre_hi;
    };

    if (CVT && warp >= 4 && warp < EW0) {
        regs_dec<kCvtRegsCvt>();
        // ----------------------- converters (CVT) -----------------------
        // warp 4 + cw converts rows 32 cw .. 32 cw + 31 of each tile; lane (g, rw)
        // = (lane / 8, lane % 8) takes row 8 G + rw of row group G and the
        // 8-index groups g and g + 4 (fp32 chunks 2g, 2g + 1 of box 0 and of box
        // 1; hi and lo chunks g and g + 4).  The eight lanes of a shared-memory
        // phase take eight rows, whose swizzled chunks differ.  Box 0 of group
        // G + 1 is loaded while group G is split.
        const int cw = warp - 4;
        const int g = lane >> 3, rw = lane & 7;
        const uint32_t ring_u = smem_u32(ring);
        Ring<NS> rr;
        bool ok = true;
        float big = 0.f;   // largest scaled magnitude (NaN if any was NaN)
        for (int64_t ty = blockIdx.y; ty < ty_end && ok; ty += ty_step) {
            const int64_t m0 = ty * kBM;
            // per-row slab scales of this warp's 32 rows (mode 0: the slab is the row)
            __syncwarp();
            if (a.slab_rows) sscale[32 * cw + lane] = y_scale_row(a, m0 + 32 * cw + lane);
            __syncwarp();
            for (int jc = jc0; jc < jc1 && ok; ++jc) {
                const int ck = chunk_len(jc);
                for (int64_t pi = pre_lo; pi < pre_hi && ok; ++pi) {
                    const float sy_pre = a.slab_rows ? 1.f : y_scale_pre(a, pi);
                    for (int q = 0; q < ck; ++q, rr.next()) {
                        if (!warp_wait_inl(&yfull[rr.slot], rr.phase, abort_flag, a.status, kStatusTimeoutLo)) {
                            ok = false;
                            break;
                        }
                        const uint32_t st = ring_u + (uint32_t)rr.slot * L::kStage;
                        // box h of row group G: this lane's two fp32 chunks (8 indices)
                        auto load = [&](int G, int h, float4* w) {
                            const uint32_t base = st + (uint32_t)h * L::kA + (uint32_t)(32 * cw + 8 * G + rw) * 128u;
                            w[0] = lds128(base + (uint32_t)(((2 * g) ^ rw) << 4));
                            w[1] = lds128(base + (uint32_t)(((2 * g + 1) ^ rw) << 4));
                        };
                        // split 8 scaled values into hi and lo words
                        auto split8 = [&](const float4* w, float sy, uint32_t* hw, uint32_t* lw) {
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float4 f = w[e >> 1];
                                const float x0 = ((e & 1) ? f.z : f.x) * sy;
                                const float x1 = ((e & 1) ? f.w : f.y) * sy;
                                big = absmax_nan(big, absmax_nan(x0, x1));
                                const __half2 hh = __floats2half2_rn(x0, x1);
                                const float2 hf = __half22float2(hh);
                                hw[e] = half2_bits(hh);
                                lw[e] = half2_bits(__floats2half2_rn(x0 - hf.x, x1 - hf.y));
                            }
                        };
                        auto put = [&](int G, int h, const uint32_t* hw, const uint32_t* lw) {
                            const uint32_t off =
                                (uint32_t)(32 * cw + 8 * G + rw) * 128u + (uint32_t)(((g + 4 * h) ^ rw) << 4);
                            sts128(st + off, hw[0], hw[1], hw[2], hw[3]);
                            sts128(st + L::kA + off, lw[0], lw[1], lw[2], lw[3]);
                        };
                        // every load of group G's rows (both boxes) precedes its stores
                        float4 a0[2], a1[2];
                        load(0, 0, a0);
#pragma unroll
                        for (int G = 0; G < 4; ++G) {
                            load(G, 1, a1);
                            const float sy = a.slab_rows ? sscale[32 * cw + 8 * G + rw] : sy_pre;
                            uint32_t hw[4], lw[4];
                            split8(a0, sy, hw, lw);
                            if (G + 1 < 4) load(G + 1, 0, a0);
                            __syncwarp();
                            put(G, 0, hw, lw);
                            split8(a1, sy, hw, lw);
                            put(G, 1, hw, lw);
                        }
                        fence_proxy_async();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&full[rr.slot]);
                    }
                }
            }
        }
        if (__any_sync(0xffffffffu, !(big < 65504.f)) && lane == 0) atomicOr(a.ovf, 1u);
    } else if (warp < 4) {
        regs_dec<CVT ? kCvtRegsCtl : kImgRegsCtl>();
        if (warp == 0 && lane == 0) {
            // ------------------------- TMA producer -------------------------
            const uint8_t* bimg = reinterpret_cast<const uint8_t*>(a.bimg);
            Ring<NS> rr;
            int64_t issued = 0;
            uint32_t nbl = 0;   // B chunks loaded so far (the B barriers' phases)
            bool ok = true;
            auto load_b = [&](int jc) -> bool {
                if (nbl > 0 && !wait_bounded_inl(bempty, (nbl - 1) & 1u, abort_flag, a.status,
                                                 kStatusTimeoutTma))
                    return false;
                const int ck = chunk_len(jc);
                mbar_arrive_expect_tx(bfull, (uint32_t)(ck * 2 * L::kB));
                for (int q = 0; q < ck; ++q) {
                    const int ks = jc * CK + q;
                    const uint8_t* src = bimg + ((int64_t)blockIdx.x * KS + ks) * (int64_t)(2 * L::kB);
                    bulk_load(bres + q * 2 * L::kB, src, 2 * L::kB, bfull);
                }
                ++nbl;
                return true;
            };
            // CVT: image coordinates of the tile in each stage, and the tiles
            // stored so far (tile u is stored once converted, from stage u % NS)
            const bool store = CVT && blockIdx.x == 0;
            int cst[CVT ? NS : 1][5];
            int64_t stored = 0;
            auto store_tile = [&](int64_t u) -> bool {
                const int sl = (int)(u % NS);
                if (!wait_bounded_inl(&full[sl], (uint32_t)((u / NS) & 1), abort_flag, a.status, kStatusTimeoutTma))
                    return false;
                const uint8_t* src = ring + sl * L::kStage;
                tma_store(&a.ymap, a.rank, cst[CVT ? sl : 0], src);
                tma_store(&a.ymap_lo, a.rank, cst[CVT ? sl : 0], src + L::kA);
                bulk_commit();
                stored = u + 1;
                return true;
            };
            // the pre index pi = (cP, cQ) in C order, advanced without divisions
            const int64_t nQ = a.nQ;
            const int cP0 = (int)(pre_lo / nQ), cQ0 = (int)(pre_lo - (int64_t)cP0 * nQ);
            for (int64_t ty = blockIdx.y; ty < ty_end && ok; ty += ty_step) {
            const int64_t m0 = ty * kBM;
            // mode-n product: (p, q) of the first row of each 64-row half
            int ttm_q0 = 0, ttm_p0 = 0, ttm_q1 = 0, ttm_p1 = 0;
            if (MN && a.ttm_q > 0) {
                ttm_p0 = (int)(m0 / a.ttm_q);
                ttm_q0 = (int)(m0 - (int64_t)ttm_p0 * a.ttm_q);
                ttm_p1 = (int)((m0 + 64) / a.ttm_q);
                ttm_q1 = (int)(m0 + 64 - (int64_t)ttm_p1 * a.ttm_q);
            }
            (void)ttm_q0; (void)ttm_p0; (void)ttm_q1; (void)ttm_p1;
            for (int jc = jc0; jc < jc1 && ok; ++jc) {
                const int ck = chunk_len(jc);
                // the first NS tiles of chunk jc need only work of chunk jc - 1,
                // so they are issued before the chunk swap
                const int64_t swap_at = issued + NS;
                bool b_pending = true;
                int cP = cP0, cQ = cQ0;
                for (int64_t pi = pre_lo; pi < pre_hi && ok; pi = unit_next(pi)) {
                    if (SMALL) {
                        cP = (int)(pi / nQ);
                        cQ = (int)(pi - (int64_t)cP * nQ);
                    }
                    for (int q = 0; q < ck; ++q, ++issued, rr.next()) {
                        // box coordinates first: they do not depend on the slot, so
                        // the copy is issued as soon as the slot is released
                        const int ks = jc * CK + q;
                        const int jp = ks / a.jq_steps;
                        int role[kRoles];
                        role[kRoleJq] = (ks - jp * a.jq_steps) * kBK4;
                        role[kRoleJp] = jp;
                        role[kRoleI] = (int)m0;
                        role[kRolePP] = cP;
                        role[kRolePQ] = cQ;
                        int c[5];
                        tma_coords(a.slot, role, c);
                        if (b_pending && issued == swap_at) {
                            b_pending = false;
                            if (!load_b(jc)) {
                                ok = false;
                                break;
                            }
                        }
                        if (rr.reused && !wait_bounded_inl(&empty[rr.slot], rr.phase ^ 1u, abort_flag,
                                                           a.status, kStatusTimeoutTma)) {
                            ok = false;
                            break;
                        }
                        if (store && rr.reused) {
                            // the stage's previous tile: stored, and its store's reads done
                            while (ok && stored <= issued - NS) ok = store_tile(stored);
                            if (!ok) break;
                            bulk_wait_read_all();
                        }
                        uint8_t* st = ring + rr.slot * L::kStage;
                        mbar_arrive_expect_tx(CVT ? &yfull[rr.slot] : &full[rr.slot], 2u * a.y_box_bytes);
                        if constexpr (CVT) {
#pragma unroll
                            for (int t = 0; t < 5; ++t) cst[rr.slot][t] = c[t];
                            // indices 0-31 of the K-step, then 32-63 (x is slot 0)
                            tma_load(&a.yfmap, a.rank, c, st, &yfull[rr.slot]);
                            c[0] += 32;
                            tma_load(&a.yfmap, a.rank, c, st + L::kA, &yfull[rr.slot]);
                            // the tile loaded NS - 1 loads ago is converted by now, or
                            // will be before the stage it holds can be refilled
                            if (store) {
                                while (ok && stored <= issued - (NS - 1)) ok = store_tile(stored);
                                if (!ok) break;
                            }
                        } else if constexpr (MN) {
                            // two 64-row halves of M per image
                            int c2[5];
                            if (a.ttm_q > 0) {
                                // mode-n product: each half is 64 consecutive q of one p
                                role[kRoleI] = ttm_q0;
                                role[kRolePP] = ttm_p0;
                                tma_coords(a.slot, role, c);
                                role[kRoleI] = ttm_q1;
                                role[kRolePP] = ttm_p1;
                            } else {
                                role[kRoleI] = (int)m0 + 64;
                            }
                            tma_coords(a.slot, role, c2);
                            tma_load(&a.ymap, a.rank, c, st, &full[rr.slot]);
                            tma_load(&a.ymap, a.rank, c2, st + L::kA / 2, &full[rr.slot]);
                            tma_load(&a.ymap_lo, a.rank, c, st + L::kA, &full[rr.slot]);
                            tma_load(&a.ymap_lo, a.rank, c2, st + L::kA + L::kA / 2, &full[rr.slot]);
                        } else {
                            tma_load(&a.ymap, a.rank, c, st, &full[rr.slot]);
                            tma_load(&a.ymap_lo, a.rank, c, st + L::kA, &full[rr.slot]);
                        }
                    }
                    if (!SMALL && ++cQ == nQ) {
                        cQ = 0;
                        ++cP;
                    }
                }
                if (ok && b_pending && !load_b(jc)) ok = false;
            }
            }   // row tiles
            if (store) {
                for (int64_t u = stored; u < issued && ok; ++u) ok = store_tile(u);
                bulk_wait_all();
            }
            for (int64_t u = issued - 1; u >= 0 && u >= issued - NS; --u)
                wait_drain_inl(CVT ? &yfull[u % NS] : &full[u % NS], (uint32_t)((u / NS) & 1), a.status);
            if (nbl > 0) wait_drain_inl(bfull, (nbl - 1) & 1u, a.status);
        } else if (warp == 1 && lane == 0) {
            // ------------------------- MMA issuer -------------------------
            // kind::f16: fp16 A and B (B K-major; A K-major, or MN-major with the
            // transpose-A bit), fp32 accumulator
            const uint32_t idesc = (1u << 4) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24) |
                                   (MN ? (1u << 15) : 0u);
            const uint32_t a_w0 = MN ? sdesc128mn_lo(smem_u32(ring)) : sdesc128_lo(smem_u32(ring));
            const uint32_t b_w0 = sdesc128_lo(smem_u32(bres));
            constexpr uint32_t kAStep = L::kStage >> 4;
            constexpr uint32_t kALo = L::kA >> 4;
            constexpr uint32_t kBStep = (2 * L::kB) >> 4;
            constexpr uint32_t kBLo = L::kB >> 4;
            Ring<NS> rr;
            int zb = 0;
            uint32_t zph = 0;
            uint32_t zused = 0;
            uint32_t nbu = 0;   // B chunks used so far
            bool ok = true;
            for (int64_t ty = blockIdx.y; ty < ty_end && ok; ty += ty_step)
            for (int jc = jc0; jc < jc1 && ok; ++jc) {
                const int ck = chunk_len(jc);
                if (!wait_bounded_inl(bfull, nbu & 1u, abort_flag, a.status, kStatusTimeoutMma)) {
                    ok = false;
                    break;
                }
                ++nbu;
                for (int64_t pi = pre_lo; pi < pre_hi && ok; pi = unit_next(pi)) {
                    uint32_t bw = b_w0;
                    for (int q = 0; q < ck; ++q, bw += kBStep, rr.next()) {
                        const bool first = q == 0;
                        const bool last = q == ck - 1;
                        if (first && ((zused >> zb) & 1u)) {
                            if (!wait_bounded_inl(&zempty[zb], (zph >> zb) & 1u, abort_flag, a.status,
                                                  kStatusTimeoutMma)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                        }
                        if (!wait_bounded_inl(&full[rr.slot], rr.phase, abort_flag, a.status, kStatusTimeoutMma)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t aw = a_w0 + (uint32_t)rr.slot * kAStep;
                        const uint32_t dz = tmem + (uint32_t)(zb * BN);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint32_t adv = (uint32_t)kk * 2u;   // 16 fp16 = 32 bytes
                            // A: 32 bytes along a K-major row, or 16 rows of 128 bytes MN-major
                            const uint32_t adva = MN ? (uint32_t)kk * 128u : adv;
                            mma_f16_ss(dz, aw + adva, bw + adv, idesc, (first && kk == 0) ? 0u : 1u);
                            mma_f16_ss(dz, aw + adva, bw + kBLo + adv, idesc, 1u);
                            mma_f16_ss(dz, aw + kALo + adva, bw + adv, idesc, 1u);
                        }
                        mma_commit(&empty[rr.slot]);
                        if (last) {
                            if (a.withhold_signal && zused == 0 && zb == 0) {
                                // test hook: this buffer is never reported full
                            } else {
                                mma_commit(&zfull[zb]);
                            }
                            if ((zused >> zb) & 1u) zph ^= 1u << zb;
                            zused |= 1u << zb;
                            zb ^= 1;
                        }
                    }
                }
                if (ok) mma_commit(bempty);
            }
            mma_commit(mma_done);
            wait_drain_inl(mma_done, 0, a.status);
        }
    } else {
        regs_inc<CVT ? kCvtRegsEpi : kImgRegsEpi>();
        // ---------------------- epilogue (16 warps) ----------------------
        constexpr int kCols = BN / 4;
        if constexpr (SMALL) {
            // TMEM lane slot * I + i holds pre index pi_u + slot of the unit; each
            // lane reads its own G row at every drain.  At the end the slots are
            // summed through shared memory.
            static_assert(kCols % kImgEpiLd == 0, "TMEM load width");
            const int quad = warp & 3;
            const int part = (warp - EW0) >> 2;
            const int64_t c0 = r0 + part * kCols;
            const int Iv = (int)a.I;
            const int lg = 32 * quad + lane;
            const int slot = lg / Iv;
            float acc[kCols];
#pragma unroll
            for (int e = 0; e < kCols; ++e) acc[e] = 0.f;
            int zb = 0;
            uint32_t zph = 0;
            bool ok = true;
            for (int jc = jc0; jc < jc1 && ok; ++jc) {
                for (int64_t pi = pre_lo; pi < pre_hi && ok; pi = unit_next(pi)) {
                    const int64_t pe = unit_next(pi);
                    const bool live_row = slot < a.ps && pi + slot < pe;
                    const float* grow = a.gtab + (pi + slot) * a.R + c0;
                    if (!warp_wait_inl(&zfull[zb], (zph >> zb) & 1u, abort_flag, a.status, kStatusTimeoutEpi)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t tbase =
                        tmem + ((uint32_t)(32 * quad) << 16) + (uint32_t)(zb * BN + part * kCols);
#pragma unroll
                    for (int cc = 0; cc < kCols; cc += kImgEpiLd) {
                        float g[kImgEpiLd];   // this row's G values for the group
#pragma unroll
                        for (int q = 0; q < kImgEpiLd; ++q)
                            g[q] = (live_row && c0 + cc + q < a.R) ? __ldg(grow + cc + q) : 0.f;
                        uint32_t z[kImgEpiLd];
                        tmem_ld_cols<kImgEpiLd>(tbase + cc, z);
                        tmem_ld_wait();
#pragma unroll
                        for (int q = 0; q < kImgEpiLd; ++q)
                            acc[cc + q] = fmaf(g[q], __uint_as_float(z[q]), acc[cc + q]);
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&zempty[zb]);
                    zph ^= 1u << zb;
                    zb ^= 1;
                }
            }
            // sum the slots: rows slot * I + i of a [128][BN + 4] buffer over the
            // (now idle) B chunk and operand stages
            constexpr int kSP = BN + 4;
            float* S = reinterpret_cast<float*>(smem);
            const bool live = !*abort_flag;
            if (live) {
#pragma unroll
                for (int e = 0; e < kCols; e += 4)
                    *reinterpret_cast<float4*>(S + lg * kSP + part * kCols + e) =
                        make_float4(acc[e], acc[e + 1], acc[e + 2], acc[e + 3]);
            }
            asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * 32) : "memory");
            if (live) {
                float* dst = a.dst + (int64_t)blockIdx.z * a.dst_split_stride;
                for (int idx = tid - 32 * EW0; idx < Iv * BN; idx += kEpiWarps * 32) {
                    const int i = idx / BN, c = idx - i * BN;
                    if (r0 + c >= a.R) continue;
                    float sum = 0.f;
                    for (int sl = 0; sl < a.ps; ++sl) sum += S[(sl * Iv + i) * kSP + c];
                    dst[(int64_t)i * a.R + r0 + c] = sum * y_unscale(a, i) * pow2_recip(a.colscale[r0 + c]);
                }
            }
        } else {
        constexpr int kGv = (kCols + 31) / 32;   // G values a lane holds
        static_assert(kCols % kImgEpiLd == 0, "TMEM load width");
        const int quad = warp & 3;
        const int part = (warp - EW0) >> 2;
        const int64_t c0 = r0 + part * kCols;
        // reciprocals of the column tile's scales, once a CTA (exact powers of two)
        for (int c = tid - 32 * EW0; c < BN; c += kEpiWarps * 32)
            colinv[c] = r0 + c < a.R ? pow2_recip(a.colscale[r0 + c]) : 0.f;
        asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * 32) : "memory");
        const float* cinv = colinv + part * kCols;
        int zb = 0;
        uint32_t zph = 0;
        bool ok = true;
        for (int64_t ty = blockIdx.y; ty < ty_end && ok; ty += ty_step) {
        const int64_t row = ty * kBM + 32 * quad + lane;
        float acc[kCols];
#pragma unroll
        for (int e = 0; e < kCols; ++e) acc[e] = 0.f;
        // G(pi, c0 + 32 u + lane) in lane `lane`, slot u; broadcast by shuffles
        auto load_g = [&](int64_t pi, float* g) {
#pragma unroll
            for (int u = 0; u < kGv; ++u) {
                const int e = 32 * u + lane;
                g[u] = (!a.g_ones && e < kCols && c0 + e < a.R && pi < pre_hi) ? __ldg(a.gtab + pi * a.R + c0 + e)
                                                                                : 0.f;
            }
        };
        float g_next[kGv];
        load_g(pre_lo, g_next);
        for (int jc = jc0; jc < jc1 && ok; ++jc) {
            for (int64_t pi = pre_lo; pi < pre_hi && ok; ++pi) {
                float g_cur[kGv];
#pragma unroll
                for (int u = 0; u < kGv; ++u) g_cur[u] = g_next[u];
                load_g(pi + 1 < pre_hi ? pi + 1 : pre_lo, g_next);   // used at the next drain
                if (!warp_wait_inl(&zfull[zb], (zph >> zb) & 1u, abort_flag, a.status, kStatusTimeoutEpi)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t tbase =
                    tmem + ((uint32_t)(32 * quad) << 16) + (uint32_t)(zb * BN + part * kCols);
#pragma unroll
                for (int cc = 0; cc < kCols; cc += kImgEpiLd) {
                    uint32_t z[kImgEpiLd];
                    tmem_ld_cols<kImgEpiLd>(tbase + cc, z);
                    tmem_ld_wait();
                    if (a.g_ones) {
#pragma unroll
                        for (int q = 0; q < kImgEpiLd; ++q) acc[cc + q] += __uint_as_float(z[q]);
                    } else {
#pragma unroll
                        for (int q = 0; q < kImgEpiLd; ++q) {
                            const int e = cc + q;
                            const float g = __shfl_sync(0xffffffffu, g_cur[e / 32], e % 32);
                            acc[e] = fmaf(g, __uint_as_float(z[q]), acc[e]);
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&zempty[zb]);
                zph ^= 1u << zb;
                zb ^= 1;
            }
        }
        if (!*abort_flag && row < a.I && a.ttm_q > 0) {
            // mode-n product: column j of row (p, q) is T[p, j, q]; the lanes of a
            // warp hold consecutive q, so each store instruction writes 128 bytes
            const float inv_y = y_unscale(a, row);
            const int64_t p = row / a.ttm_q, q = row - p * a.ttm_q;
            float* dst = a.dst + p * a.R * a.ttm_q + q;
#pragma unroll
            for (int e = 0; e < kCols; ++e)
                if (c0 + e < a.R) dst[(c0 + e) * a.ttm_q] = acc[e] * inv_y * cinv[e];
        } else if (!*abort_flag && row < a.I) {
            // undo the power-of-two scales of Y and of each Binner column (exact)
            const float inv_y = y_unscale(a, row);
            float* dst = a.dst + (int64_t)blockIdx.z * a.dst_split_stride + row * a.R + c0;
            const bool vst = (a.R % 4 == 0) && ((reinterpret_cast<uintptr_t>(a.dst) & 15) == 0);
#pragma unroll
            for (int e = 0; e < kCols; e += 4) {
                const float4 ci = *reinterpret_cast<const float4*>(cinv + e);
                const float v[4] = {acc[e] * inv_y * ci.x, acc[e + 1] * inv_y * ci.y, acc[e + 2] * inv_y * ci.z,
                                    acc[e + 3] * inv_y * ci.w};
                if (vst && c0 + e + 4 <= a.R) {
                    *reinterpret_cast<float4*>(dst + e) = make_float4(v[0], v[1], v[2], v[3]);
                } else {
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        if (c0 + e + q < a.R) dst[e + q] = v[q];
                }
            }
        }
        }   // row tiles
        }   // not SMALL
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
    }
}

// Work units of the passes over Y that need a slab's scale: at most kSlabUnit
// consecutive elements of one slab of mode 0 (nslab slabs of len elements; one
// slab when the plan scales Y as a whole).  A block takes a contiguous run of
// units, so it meets each slab in one stretch.
constexpr int kSlabUnit = 8192;

struct SlabUnits {
    int64_t ups, u0, u1;   // units per slab, this block's units [u0, u1)
    __device__ SlabUnits(int64_t nslab, int64_t len) {
        ups = (len + kSlabUnit - 1) / kSlabUnit;
        const int64_t n = nslab * ups;
        const int64_t per = (n + gridDim.x - 1) / gridDim.x;
        u0 = (int64_t)blockIdx.x * per;
        u1 = u0 + per < n ? u0 + per : n;
    }
};

// Split Y into the fp16 images the kernel above streams: with x = Y * s (s the
// power of two of Y's slab of mode 0), hi = fp16(x) and lo = fp16(x - hi) (the
// difference is exact in fp32), same layout as Y.  Units as in slabmax_kernel.
__device__ __forceinline__ void split1(float v, float sy, __half& h, __half& l) {
    const float x = v * sy;
    h = __float2half_rn(x);
    l = __float2half_rn(x - __half2float(h));
}

// With ovf non-null, a scaled value outside the fp16 range (|x| >= 65504, or
// not a number) sets *ovf: the scales came from sampled maxima that missed a
// larger entry, and the exact pass that follows redoes maxima and images.  With
// enable non-null the kernel runs only if *enable is set (that exact pass).
__device__ __forceinline__ bool fp16_out_of_range(float x) { return !(fabsf(x) < 65504.f); }

__global__ void __launch_bounds__(256) split_image_kernel(const float* __restrict__ y, int64_t nslab, int64_t len,
                                                          const uint32_t* __restrict__ slab,
                                                          const uint32_t* __restrict__ gmax,
                                                          __half* __restrict__ hi, __half* __restrict__ lo,
                                                          uint32_t* __restrict__ ovf,
                                                          const uint32_t* __restrict__ enable) {
    if (enable != nullptr && *enable == 0) return;
    const SlabUnits su(nslab, len);
    const uint32_t gbits = *gmax;
    bool bad = false;
    // y, hi and lo 16-byte aligned (the images are): whole units move as float4
    const bool vec = (len % 4 == 0) && (reinterpret_cast<uintptr_t>(y) & 15) == 0;
    for (int64_t u = su.u0; u < su.u1; ++u) {
        const int64_t s = u / su.ups;
        const float sy = slab_scale(slab, s, gbits);
        const int64_t a0 = s * len + (u - s * su.ups) * kSlabUnit;
        const int64_t a1 = min(a0 + kSlabUnit, (s + 1) * len);
        if (vec && a1 - a0 == kSlabUnit) {
            const int64_t f0 = a0 / 4 + threadIdx.x;
            float4 v[kSlabUnit / 1024];
#pragma unroll
            for (int q = 0; q < kSlabUnit / 1024; ++q) v[q] = __ldcs(reinterpret_cast<const float4*>(y) + f0 + 256 * q);
#pragma unroll
            for (int q = 0; q < kSlabUnit / 1024; ++q) {
                const float x0 = v[q].x * sy, x1 = v[q].y * sy, x2 = v[q].z * sy, x3 = v[q].w * sy;
                bad |= fp16_out_of_range(fmaxf(fmaxf(fabsf(x0), fabsf(x1)), fmaxf(fabsf(x2), fabsf(x3)))) ||
                       x0 != x0 || x1 != x1 || x2 != x2 || x3 != x3;
                const __half2 h01 = __floats2half2_rn(x0, x1), h23 = __floats2half2_rn(x2, x3);
                const float2 f01 = __half22float2(h01), f23 = __half22float2(h23);
                const __half2 l01 = __floats2half2_rn(x0 - f01.x, x1 - f01.y);
                const __half2 l23 = __floats2half2_rn(x2 - f23.x, x3 - f23.y);
                reinterpret_cast<uint2*>(hi)[f0 + 256 * q] = make_uint2(half2_bits(h01), half2_bits(h23));
                reinterpret_cast<uint2*>(lo)[f0 + 256 * q] = make_uint2(half2_bits(l01), half2_bits(l23));
            }
        } else {
            for (int64_t i = a0 + threadIdx.x; i < a1; i += blockDim.x) {
                const float v = __ldcs(y + i);
                bad |= fp16_out_of_range(v * sy);
                split1(v, sy, hi[i], lo[i]);
            }
        }
    }
    if (ovf != nullptr && __syncthreads_or(bad) && threadIdx.x == 0) atomicOr(ovf, 1u);
}

// The same split for the innermost mode: Y viewed as P x I (I = I_{d-1}, the
// contiguous mode) is also written transposed, I x P, so that the innermost
// mode's tiles are K-contiguous too.  One 64 (p) x 128 (i) tile per step: each
// warp reads rows of 128 consecutive i (16-byte loads; scalar when I is not a
// multiple of 4), converts, optionally writes the natural images (8-byte
// stores), and parks (hi | lo << 16) in shared memory; then each warp writes
// rows of 64 consecutive p of both transposed images (4-byte stores, P even).
// Rows p of the P x I view belong to slab p / rps of mode 0 (rps rows a slab).
template <bool VEC>
__global__ void __launch_bounds__(256, 3) split_image_t_kernel(const float* __restrict__ y, int64_t P, int64_t I,
                                                            const uint32_t* __restrict__ slab,
                                                            const uint32_t* __restrict__ gmax, int64_t rps,
                                                            __half* __restrict__ hi, __half* __restrict__ lo,
                                                            __half* __restrict__ thi, __half* __restrict__ tlo,
                                                            int write_nat, uint32_t* __restrict__ ovf,
                                                            const uint32_t* __restrict__ enable) {
    if (enable != nullptr && *enable == 0) return;
    bool bad = false;
    constexpr int TP = 64, TI = 128;
    __shared__ uint32_t sh[TI][TP + 1];   // [i][p]: hi in the low half, lo in the high half
    const uint32_t gbits = *gmax;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // scale of row pr of the tile starting at row p0: a tile of TP rows meets at
    // most two slabs when a slab has at least TP rows
    int64_t s_b1 = 0;
    float s_sy0 = 1.f, s_sy1 = 1.f;
    auto tile_scales = [&](int64_t p0) {
        const int64_t s0 = p0 / rps;
        s_b1 = (s0 + 1) * rps;
        s_sy0 = slab_scale(slab, s0, gbits);
        s_sy1 = s_b1 < P ? slab_scale(slab, s0 + 1, gbits) : s_sy0;
    };
    auto row_scale = [&](int64_t pr, int64_t tile_rows) -> float {   // rows past P clamp to the last
        return rps >= tile_rows ? (pr >= s_b1 ? s_sy1 : s_sy0)
                                : slab_scale(slab, (pr < P ? pr : P - 1) / rps, gbits);
    };
    if (I < TI / 2) {
        // short rows: TPS consecutive p (as many as the shared array holds, a
        // multiple of 64) are one contiguous block of TPS * I values, read (and
        // written in the natural layout) flat, so that no lanes idle; staged as
        // [i][p] with a row stride of TPS + 1 words
        const int Ii = (int)I;
        int tps = (TI * (TP + 1)) / Ii - 1;
        tps = tps >= 1024 ? 1024 : (tps / TP) * TP;
        const int stride = tps + 1;
        uint32_t* shf = &sh[0][0];
        const int64_t np = (P + tps - 1) / tps;
        for (int64_t t = blockIdx.x; t < np; t += gridDim.x) {
            const int64_t p0 = t * tps;
            const int rows = (int)(P - p0 < tps ? P - p0 : tps);
            tile_scales(p0);
            const int nvals = rows * Ii;
            const int64_t base = p0 * I;
            // four 16-byte loads in flight a thread before any conversion; the
            // (row, col) of a thread's value 4 f is stepped from one division
            constexpr int kU = 4;
            const int step_r = (4 * 256) / Ii, step_c = (4 * 256) - step_r * Ii;   // 4 * 256 values
            int row0 = (4 * (int)threadIdx.x) / Ii;
            int col0 = 4 * (int)threadIdx.x - row0 * Ii;
            for (int f0 = 0; 4 * f0 < nvals; f0 += kU * 256) {
                float4 vv[kU];
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int f = f0 + threadIdx.x + 256 * u;
                    vv[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (4 * f + 3 < nvals) {
                        vv[u] = __ldcs(reinterpret_cast<const float4*>(y + base) + f);
                    } else if (4 * f < nvals) {
                        float t[4] = {0.f, 0.f, 0.f, 0.f};
                        for (int q = 0; q < 4; ++q)
                            if (4 * f + q < nvals) t[q] = __ldcs(y + base + 4 * f + q);
                        vv[u] = make_float4(t[0], t[1], t[2], t[3]);
                    }
                }
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int f = f0 + threadIdx.x + 256 * u;
                    int row = row0, col = col0;   // (row, col) of value 4 f
                    row0 += step_r;
                    col0 += step_c;
                    if (col0 >= Ii) {
                        col0 -= Ii;
                        ++row0;
                    }
                    if (4 * f >= nvals) continue;
                    const float v[4] = {vv[u].x, vv[u].y, vv[u].z, vv[u].w};
                    uint32_t hb[4], lb[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int idx = 4 * f + q;
                        const float x = v[q] * row_scale(p0 + row, tps);
                        bad |= fp16_out_of_range(x);
                        const __half h = __float2half_rn(x);
                        const __half l = __float2half_rn(x - __half2float(h));
                        hb[q] = __half_as_ushort(h);
                        lb[q] = __half_as_ushort(l);
                        if (idx < nvals) shf[col * stride + row] = hb[q] | (lb[q] << 16);
                        if (++col == Ii) {
                            col = 0;
                            ++row;
                        }
                    }
                    if (write_nat) {
                        if (4 * f + 3 < nvals) {
                            reinterpret_cast<uint2*>(hi + base)[f] =
                                make_uint2(hb[0] | (hb[1] << 16), hb[2] | (hb[3] << 16));
                            reinterpret_cast<uint2*>(lo + base)[f] =
                                make_uint2(lb[0] | (lb[1] << 16), lb[2] | (lb[3] << 16));
                        } else {
                            for (int q = 0; q < 4; ++q)
                                if (4 * f + q < nvals) {
                                    hi[base + 4 * f + q] = __ushort_as_half((unsigned short)hb[q]);
                                    lo[base + 4 * f + q] = __ushort_as_half((unsigned short)lb[q]);
                                }
                        }
                    }
                }
            }
            __syncthreads();
            // transposed: row c holds p0 .. p0 + rows - 1 at c * P + p, two p a lane;
            // (c, pair) of item w stepped from one division
            const int pairs = (rows + 1) / 2;
            const int sc = (int)blockDim.x / pairs, sp = (int)blockDim.x - sc * pairs;
            int c_w = (int)threadIdx.x / pairs, p_w = (int)threadIdx.x - c_w * pairs;
            for (int w = threadIdx.x; w < Ii * pairs; w += blockDim.x) {
                const int c = c_w, pp = 2 * p_w;
                c_w += sc;
                p_w += sp;
                if (p_w >= pairs) {
                    p_w -= pairs;
                    ++c_w;
                }
                const uint32_t w0 = shf[c * stride + pp];
                const int64_t e = (int64_t)c * P + p0 + pp;
                if (pp + 1 < rows) {
                    const uint32_t w1 = shf[c * stride + pp + 1];
                    *reinterpret_cast<uint32_t*>(thi + e) = __byte_perm(w0, w1, 0x5410);
                    *reinterpret_cast<uint32_t*>(tlo + e) = __byte_perm(w0, w1, 0x7632);
                } else {
                    thi[e] = __ushort_as_half((unsigned short)(w0 & 0xFFFFu));
                    tlo[e] = __ushort_as_half((unsigned short)(w0 >> 16));
                }
            }
            __syncthreads();
        }
        if (ovf != nullptr && __syncthreads_or(bad) && threadIdx.x == 0) atomicOr(ovf, 1u);
        return;
    }
    const int64_t np = (P + TP - 1) / TP, ni = (I + TI - 1) / TI;
    for (int64_t t = blockIdx.x; t < np * ni; t += gridDim.x) {
        const int64_t p0 = (t / ni) * TP, i0 = (t % ni) * TI;
        const int64_t ib = i0 + 4 * lane;   // this lane's first i
        tile_scales(p0);
        // all eight rows' loads first (eight 16-byte loads in flight a thread)
        float vv[TP / 8][4];
#pragma unroll
        for (int u = 0; u < TP / 8; ++u) {
            const int64_t pr = p0 + warp + 8 * u;
            const int64_t e = pr * I + ib;
#pragma unroll
            for (int q = 0; q < 4; ++q) vv[u][q] = 0.f;
            if (pr < P) {
                if (VEC) {
                    if (ib < I) {
                        const float4 x = __ldcs(reinterpret_cast<const float4*>(y + e));
                        vv[u][0] = x.x;
                        vv[u][1] = x.y;
                        vv[u][2] = x.z;
                        vv[u][3] = x.w;
                    }
                } else {
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        if (ib + q < I) vv[u][q] = __ldcs(y + e + q);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < TP / 8; ++u) {
            const int r = warp + 8 * u;
            const int64_t pr = p0 + r;
            const int64_t e = pr * I + ib;
            const float* v = vv[u];
            const float sy = row_scale(pr, TP);
            uint32_t hb[4], lb[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float x = v[q] * sy;
                bad |= fp16_out_of_range(x);
                const __half h = __float2half_rn(x);
                const __half l = __float2half_rn(x - __half2float(h));
                hb[q] = __half_as_ushort(h);
                lb[q] = __half_as_ushort(l);
                sh[4 * lane + q][r] = hb[q] | (lb[q] << 16);
            }
            if (write_nat && pr < P) {
                if (VEC) {
                    if (ib < I) {
                        reinterpret_cast<uint2*>(hi + e)[0] = make_uint2(hb[0] | (hb[1] << 16), hb[2] | (hb[3] << 16));
                        reinterpret_cast<uint2*>(lo + e)[0] = make_uint2(lb[0] | (lb[1] << 16), lb[2] | (lb[3] << 16));
                    }
                } else {
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        if (ib + q < I) {
                            hi[e + q] = __ushort_as_half((unsigned short)hb[q]);
                            lo[e + q] = __ushort_as_half((unsigned short)lb[q]);
                        }
                }
            }
        }
        __syncthreads();
        for (int c = warp; c < TI; c += 8) {
            const int64_t ic = i0 + c;
            const int64_t pc = p0 + 2 * lane;
            if (ic < I && pc < P) {
                const uint32_t w0 = sh[c][2 * lane], w1 = sh[c][2 * lane + 1];
                const int64_t e = ic * P + pc;
                if (pc + 1 < P) {
                    *reinterpret_cast<uint32_t*>(thi + e) = __byte_perm(w0, w1, 0x5410);
                    *reinterpret_cast<uint32_t*>(tlo + e) = __byte_perm(w0, w1, 0x7632);
                } else {
                    thi[e] = __ushort_as_half((unsigned short)(w0 & 0xFFFFu));
                    tlo[e] = __ushort_as_half((unsigned short)(w0 >> 16));
                }
            }
        }
        __syncthreads();
    }
    if (ovf != nullptr && __syncthreads_or(bad) && threadIdx.x == 0) atomicOr(ovf, 1u);
}

// ---------------------------------------------------------------------------
// Prep: pre-swizzled hi/lo images of the inner Khatri-Rao table
// ---------------------------------------------------------------------------

struct BImgArgs {
    int ngroup;
    int64_t gdim[kMaxD];
    const float* gfac[kMaxD];
    int64_t R, J, Jq;
    int BN, KS, jq_steps, inner;
    int64_t nblocks;   // n-tiles x KS
    float* out;
};

__global__ void tc_bimage_kernel(BImgArgs a) {
    const int64_t per_block = 2LL * a.BN * kBK;  // floats (hi + lo)
    const int64_t n = a.nblocks * per_block;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t blk = e / per_block;
        const int64_t w = e - blk * per_block;
        const int half = (int)(w / (a.BN * kBK));
        const int64_t w2 = w - (int64_t)half * a.BN * kBK;
        const uint32_t byte = (uint32_t)(w2 * 4);
        const uint32_t row = byte / 64u;
        const uint32_t chunk_pos = (byte % 64u) / 16u;
        const uint32_t elem = (byte % 16u) / 4u;
        const uint32_t kk = ((chunk_pos ^ (row >> 1)) & 3u) * 4u + elem;
        const int64_t nt = blk / a.KS;
        const int ks = (int)(blk - nt * a.KS);
        const int64_t r = nt * a.BN + row;
        int64_t j;
        bool valid;
        if (a.inner) {
            j = (int64_t)ks * kBK + kk;
            valid = j < a.J;
        } else {
            const int jp = ks / a.jq_steps;
            const int64_t jq = (int64_t)(ks - jp * a.jq_steps) * kBK + kk;
            valid = jq < a.Jq;
            j = (int64_t)jp * a.Jq + jq;
        }
        float v = 0.f;
        if (valid && r < a.R) {
            int64_t rem = j;
            v = 1.f;
            for (int m = a.ngroup - 1; m >= 0; --m) {
                const int64_t idx = rem % a.gdim[m];
                rem /= a.gdim[m];
                v *= a.gfac[m][idx * a.R + r];
            }
        }
        a.out[e] = half == 0 ? v : v - __uint_as_float(__float_as_uint(v) & kTf32Mask);
    }
}

// Largest magnitude of every slab of mode 0 (slab[s]) and of the whole tensor
// (*gmax), as fp32 bits (non-negative floats order like their bits).  Each block
// flushes its running maximum with one atomicMax per slab it touches and one on
// *gmax at the end.  slab[] and *gmax must be zero, or hold lower bounds of the
// maxima (the sampled ones), before the launch.  With enable non-null the
// kernel runs only if *enable is set.
__global__ void __launch_bounds__(256) slabmax_kernel(const float* __restrict__ y, int64_t nslab, int64_t len,
                                                      uint32_t* __restrict__ slab, uint32_t* __restrict__ gmax,
                                                      const uint32_t* __restrict__ enable) {
    if (enable != nullptr && *enable == 0) return;
    __shared__ uint32_t wm[8];
    const SlabUnits su(nslab, len);
    const bool vec = (len % 4 == 0) && (reinterpret_cast<uintptr_t>(y) & 15) == 0;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t m = 0, g = 0;
    auto block_max = [&](uint32_t v) -> uint32_t {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
        if (lane == 0) wm[warp] = v;
        __syncthreads();
        uint32_t r = wm[0];
#pragma unroll
        for (int w = 1; w < 8; ++w) r = max(r, wm[w]);
        __syncthreads();
        return r;
    };
    int64_t cur = -1;
    for (int64_t u = su.u0; u < su.u1; ++u) {
        const int64_t s = u / su.ups;   // the same for every thread of the block
        if (s != cur) {
            if (cur >= 0) {
                const uint32_t b = block_max(m);
                if (threadIdx.x == 0 && b) atomicMax(slab + cur, b);
                g = max(g, b);
            }
            m = 0;
            cur = s;
        }
        const int64_t a0 = s * len + (u - s * su.ups) * kSlabUnit;
        const int64_t a1 = min(a0 + kSlabUnit, (s + 1) * len);
        if (vec && a1 - a0 == kSlabUnit) {
            // a whole unit: eight 16-byte loads in flight a thread
            const float4* p = reinterpret_cast<const float4*>(y + a0) + threadIdx.x;
            float4 v[kSlabUnit / 1024];
#pragma unroll
            for (int q = 0; q < kSlabUnit / 1024; ++q) v[q] = __ldcs(p + 256 * q);
#pragma unroll
            for (int q = 0; q < kSlabUnit / 1024; ++q) {
                m = max(m, __float_as_uint(fabsf(v[q].x)));
                m = max(m, __float_as_uint(fabsf(v[q].y)));
                m = max(m, __float_as_uint(fabsf(v[q].z)));
                m = max(m, __float_as_uint(fabsf(v[q].w)));
            }
        } else {
            for (int64_t i = a0 + threadIdx.x; i < a1; i += blockDim.x) m = max(m, __float_as_uint(fabsf(y[i])));
        }
    }
    if (cur >= 0) {
        const uint32_t b = block_max(m);
        if (threadIdx.x == 0 && b) atomicMax(slab + cur, b);
        g = max(g, b);
    }
    if (threadIdx.x == 0 && g) atomicMax(gmax, g);
}

// Sampled maxima: every kSampleEvery-th chunk of kSampleChunk consecutive
// elements of each slab (all of a slab of at most kSampleEvery chunks), a lower
// bound of the slab's largest magnitude, stored (atomicMax) as at least the
// smallest subnormal's bits, so that no sampled slab reads as all-zero: a scale
// from a lower bound is at least the exact one (every value keeps at least the
// exact path's precision), and a value it pushes out of the fp16 range is caught
// by the split (which then calls for the exact maxima and images).  A warp takes
// a chunk; one atomicMax on *gmax a block.  slab[] and *gmax zero before.
constexpr int64_t kSampleChunk = 512, kSampleEvery = 16;

__global__ void __launch_bounds__(256) slabsample_kernel(const float* __restrict__ y, int64_t nslab, int64_t len,
                                                         uint32_t* __restrict__ slab, uint32_t* __restrict__ gmax) {
    __shared__ uint32_t wm[8];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t nch = (len + kSampleChunk - 1) / kSampleChunk;   // chunks a slab
    const int64_t every = nch > kSampleEvery ? kSampleEvery : 1;
    const int64_t per = (nch + every - 1) / every;                 // sampled chunks a slab
    const int64_t total = nslab * per;
    const bool vec = (len % 4 == 0) && (reinterpret_cast<uintptr_t>(y) & 15) == 0;
    uint32_t bm = 0;
    for (int64_t w = (int64_t)blockIdx.x * 8 + warp; w < total; w += (int64_t)gridDim.x * 8) {
        const int64_t s = w / per, c = (w - s * per) * every;
        const int64_t a0 = s * len + c * kSampleChunk;
        const int64_t a1 = min(a0 + kSampleChunk, (s + 1) * len);
        uint32_t m = 0;
        if (vec && a1 - a0 == kSampleChunk) {
            const float4* p = reinterpret_cast<const float4*>(y + a0) + lane;
            float4 v[kSampleChunk / 128];
#pragma unroll
            for (int q = 0; q < kSampleChunk / 128; ++q) v[q] = __ldcs(p + 32 * q);
#pragma unroll
            for (int q = 0; q < kSampleChunk / 128; ++q)
                m = max(m, max(max(__float_as_uint(fabsf(v[q].x)), __float_as_uint(fabsf(v[q].y))),
                               max(__float_as_uint(fabsf(v[q].z)), __float_as_uint(fabsf(v[q].w)))));
        } else {
            for (int64_t i = a0 + lane; i < a1; i += 32) m = max(m, __float_as_uint(fabsf(y[i])));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
        m = m > 0u ? m : 1u;
        if (lane == 0) atomicMax(slab + s, m);
        bm = max(bm, m);
    }
    if (lane == 0) wm[warp] = bm;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t t = 0;
        for (int q = 0; q < 8; ++q) t = max(t, wm[q]);
        if (t) atomicMax(gmax, t);
    }
}

// Power-of-two scale of each Binner column: max_j |Binner(j, r)| is the product
// over the group's modes of max_i |A_n(i, r)|; the scale maps it into
// [2^13, 2^14) (1 for a zero or non-finite column).
struct ColScaleArgs {
    int ngroup;
    int64_t gdim[kMaxD];
    const float* gfac[kMaxD];
    int64_t R;
    float* out;
};

// one block per 32 columns: 8 row groups x 32 columns, reduced through shared memory
__global__ void __launch_bounds__(1024) colscale_kernel(ColScaleArgs a) {
    __shared__ float red[32][33];
    const int lc = threadIdx.x & 31, lr = threadIdx.x >> 5;
    const int64_t r = (int64_t)blockIdx.x * 32 + lc;
    float prod = 1.f;
    for (int t = 0; t < a.ngroup; ++t) {
        float m = 0.f;
        if (r < a.R) {
#pragma unroll 4
            for (int64_t i = lr; i < a.gdim[t]; i += 32) m = fmaxf(m, fabsf(a.gfac[t][i * a.R + r]));
        }
        red[lr][lc] = m;
        __syncthreads();
        if (lr == 0) {
            for (int q = 1; q < 32; ++q) m = fmaxf(m, red[q][lc]);
            prod *= m;
        }
        __syncthreads();
    }
    if (lr == 0 && r < a.R) a.out[r] = pow2_scale(__float_as_uint(prod));
}

// fp16 hi|lo images of the scaled inner KRP table for the two-term fp16 split:
// per (n-tile, K-step of KW): hi image [BN rows][KW fp16] then lo image.
// KW = 32: rows of 64 bytes, 64-byte swizzled (16-byte chunk c of row n at
// (c ^ (n >> 1)) & 3); KW = 64: rows of 128 bytes, 128-byte swizzled (chunk c
// at (c ^ n) & 7).
template <int KW>
__global__ void tc_bimage_f16_kernel(BImgArgs a, const float* __restrict__ colscale) {
    static_assert(KW == 32 || KW == 64, "64- or 128-byte rows");
    constexpr uint32_t kRow = 2 * KW;                 // bytes per row
    const int per_block = 2 * a.BN * KW;              // fp16 elements (hi + lo)
    const int64_t n = a.nblocks * per_block;
    __half* out = reinterpret_cast<__half*>(a.out);
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t blk = e / per_block;
        const uint32_t w = (uint32_t)(e - blk * per_block);
        const uint32_t half = w / (uint32_t)(a.BN * KW);
        const uint32_t byte = (w - half * (uint32_t)(a.BN * KW)) * 2u;
        const uint32_t row = byte / kRow;
        const uint32_t chunk_pos = (byte % kRow) / 16u;
        const uint32_t elem = (byte % 16u) / 2u;
        const uint32_t kk = (KW == 32 ? ((chunk_pos ^ (row >> 1)) & 3u) : ((chunk_pos ^ row) & 7u)) * 8u + elem;
        const int64_t nt = blk / a.KS;
        const int ks = (int)(blk - nt * a.KS);
        const int64_t r = nt * a.BN + row;
        int64_t j;
        bool valid;
        if (a.inner) {
            j = (int64_t)ks * KW + kk;
            valid = j < a.J;
        } else {
            const int jp = ks / a.jq_steps;
            const int64_t jq = (int64_t)(ks - jp * a.jq_steps) * KW + kk;
            valid = jq < a.Jq;
            j = (int64_t)jp * a.Jq + jq;
        }
        float v = 0.f;
        if (valid && r < a.R) {
            v = colscale[r];
            if (a.ngroup == 1) {
                v *= a.gfac[0][j * a.R + r];   // the group's only mode: j is its index
            } else {
                int64_t rem = j;
                for (int m = a.ngroup - 1; m >= 0; --m) {
                    const int64_t idx = rem % a.gdim[m];
                    rem /= a.gdim[m];
                    v *= a.gfac[m][idx * a.R + r];
                }
            }
        }
        const __half h = __float2half_rn(v);
        out[e] = half == 0 ? h : __float2half_rn(v - __half2float(h));
    }
}

// The same images built 32 rows (columns r) of one (n-tile, K-step) block at a
// time: the KW x 32 values are formed in shared memory with the columns r
// fastest (coalesced reads of the column scales and the group factors), then
// each thread writes one 16-byte chunk of 8 values of a row of both images in
// its swizzled place.  Grid: image blocks x (BN / 32) row groups.
constexpr int kBimgRows = 32;

template <int KW>
__global__ void __launch_bounds__(256) tc_bimage_f16_tile_kernel(BImgArgs a, const float* __restrict__ colscale) {
    static_assert(KW == 32 || KW == 64, "64- or 128-byte rows");
    constexpr int kChunks = KW / 8;
    constexpr int S = kBimgRows + 1;
    __shared__ float vs[KW * S];   // [kk][row in the group]
    const int BN = a.BN;
    const int groups = BN / kBimgRows;
    const int64_t total = a.nblocks * groups;
    for (int64_t t = blockIdx.x; t < total; t += gridDim.x) {
        const int64_t blk = t / groups;
        const int rg = (int)(t - blk * groups);
        const int64_t nt = blk / a.KS;
        const int ks = (int)(blk - nt * a.KS);
        for (int e = threadIdx.x; e < KW * kBimgRows; e += blockDim.x) {
            const int kk = e / kBimgRows, rl = e - kk * kBimgRows;
            const int64_t r = nt * BN + rg * kBimgRows + rl;
            int64_t j;
            bool valid;
            if (a.inner) {
                j = (int64_t)ks * KW + kk;
                valid = j < a.J;
            } else {
                const int jp = ks / a.jq_steps;
                const int64_t jq = (int64_t)(ks - jp * a.jq_steps) * KW + kk;
                valid = jq < a.Jq;
                j = (int64_t)jp * a.Jq + jq;
            }
            float v = 0.f;
            if (valid && r < a.R) {
                v = colscale[r];
                if (a.ngroup == 1) {
                    v *= a.gfac[0][j * a.R + r];
                } else {
                    int64_t rem = j;
                    for (int m = a.ngroup - 1; m >= 0; --m) {
                        const int64_t idx = rem % a.gdim[m];
                        rem /= a.gdim[m];
                        v *= a.gfac[m][idx * a.R + r];
                    }
                }
            }
            vs[kk * S + rl] = v;
        }
        __syncthreads();
        __half* out = reinterpret_cast<__half*>(a.out) + blk * (int64_t)(2 * BN * KW);
        for (int w = threadIdx.x; w < kBimgRows * kChunks; w += blockDim.x) {
            const int rl = w / kChunks, c = w - rl * kChunks;
            const int rr = rg * kBimgRows + rl;
            uint32_t hw[4], lw[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float v0 = vs[(8 * c + 2 * q) * S + rl], v1 = vs[(8 * c + 2 * q + 1) * S + rl];
                const __half h0 = __float2half_rn(v0), h1 = __float2half_rn(v1);
                const __half l0 = __float2half_rn(v0 - __half2float(h0)), l1 = __float2half_rn(v1 - __half2float(h1));
                hw[q] = (uint32_t)__half_as_ushort(h0) | ((uint32_t)__half_as_ushort(h1) << 16);
                lw[q] = (uint32_t)__half_as_ushort(l0) | ((uint32_t)__half_as_ushort(l1) << 16);
            }
            const int pos = KW == 32 ? ((c ^ (rr >> 1)) & 3) : ((c ^ rr) & 7);
            *reinterpret_cast<uint4*>(out + (int64_t)rr * KW + pos * 8) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            *reinterpret_cast<uint4*>(out + (int64_t)BN * KW + (int64_t)rr * KW + pos * 8) =
                make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
        __syncthreads();
    }
}

// launch helper: the tile kernel for tiles of whole 32-row groups, else the
// element-wise one
template <int KW>
cudaError_t launch_bimage_f16(const BImgArgs& b, const float* colscale, cudaStream_t stream) {
    if (b.BN % kBimgRows == 0 && (reinterpret_cast<uintptr_t>(b.out) & 15) == 0) {
        int64_t blocks = b.nblocks * (b.BN / kBimgRows);
        if (blocks > 152 * 8) blocks = 152 * 8;
        tc_bimage_f16_tile_kernel<KW><<<(unsigned)(blocks > 0 ? blocks : 1), 256, 0, stream>>>(b, colscale);
        return cudaGetLastError();
    }
    int64_t blocks = (b.nblocks * 2 * b.BN * KW + 255) / 256;
    if (blocks > 152 * 16) blocks = 152 * 16;
    tc_bimage_f16_kernel<KW><<<(unsigned)blocks, 256, 0, stream>>>(b, colscale);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// The explicit Khatri-Rao product (matrix-based comparison variant), written
// as the B images the tensor-core kernels stream: row j of the product (j over
// every mode but k, C order) is KRP(j, r) = T1(j / I_last, r) * A_last(j % I_last, r),
// T1 being the product of the other group factors (a table built beforehand).
// One block of the images per (column tile nt, K-step ks): the KW rows j of the
// K-step are decoded once, the KW x BN values staged in shared memory (columns
// r fastest, so the table and factor reads are coalesced), then written as hi
// and lo images in the swizzled layout of the kernel that reads them:
//   F16  (fp16-image kernel): KW = 64, 128-byte rows, chunk c of row n at
//        (c ^ n) & 7, values scaled by the column's power of two,
//        hi = fp16(v), lo = fp16(v - hi);
//   fp32 (3xTF32 kernel):     KW = 16, 64-byte rows, chunk c of row n at
//        (c ^ (n >> 1)) & 3, hi = v (the tensor core truncates it to tf32),
//        lo = v - tf32(v).
// ---------------------------------------------------------------------------
struct KrpImgArgs {
    const float* t1;        // (J / I_last) x R
    const float* alast;     // I_last x R
    int64_t ilast;
    const float* colscale;  // R (F16 only)
    int64_t R, J, Jq;
    int BN, KS, jq_steps, inner;
    int64_t nblocks;        // column tiles x KS
    void* out;
};

constexpr int kKrpMaxBN = 256;

template <int KW, bool F16>
__global__ void __launch_bounds__(256) krp_image_kernel(KrpImgArgs a) {
    extern __shared__ float vs[];           // [KW][BN]
    __shared__ int64_t jrow1[KW], jrow2[KW];   // j / I_last and j % I_last, -1: padding
    constexpr int kChunk = 16 / (F16 ? 2 : 4);     // values a 16-byte chunk holds
    constexpr int kChunks = KW / kChunk;           // chunks a row
    constexpr int kRow = KW * (F16 ? 2 : 4);       // bytes a row
    const int BN = a.BN;
    for (int64_t blk = blockIdx.x; blk < a.nblocks; blk += gridDim.x) {
        const int64_t nt = blk / a.KS;
        const int ks = (int)(blk - nt * a.KS);
        if (threadIdx.x < KW) {
            const int kk = threadIdx.x;
            int64_t j;
            bool valid;
            if (a.inner) {
                j = (int64_t)ks * KW + kk;
                valid = j < a.J;
            } else {
                const int jp = ks / a.jq_steps;
                const int64_t jq = (int64_t)(ks - jp * a.jq_steps) * KW + kk;
                valid = jq < a.Jq;
                j = (int64_t)jp * a.Jq + jq;
            }
            jrow1[kk] = valid ? j / a.ilast : -1;
            jrow2[kk] = valid ? j - (j / a.ilast) * a.ilast : 0;
        }
        __syncthreads();
        for (int e = threadIdx.x; e < KW * BN; e += blockDim.x) {
            const int kk = e / BN, c = e - kk * BN;
            const int64_t r = nt * BN + c;
            float v = 0.f;
            if (jrow1[kk] >= 0 && r < a.R) {
                v = __ldg(a.t1 + jrow1[kk] * a.R + r) * __ldg(a.alast + jrow2[kk] * a.R + r);
                if constexpr (F16) v *= __ldg(a.colscale + r);
            }
            vs[e] = v;
        }
        __syncthreads();
        uint8_t* base = static_cast<uint8_t*>(a.out) + blk * (int64_t)(2 * BN * kRow);
        for (int t = threadIdx.x; t < BN * kChunks; t += blockDim.x) {
            const int n = t / kChunks, cp = t - n * kChunks;
            const int lc = F16 ? ((cp ^ n) & 7) : ((cp ^ (n >> 1)) & 3);   // logical chunk held at cp
            float v[kChunk];
#pragma unroll
            for (int q = 0; q < kChunk; ++q) v[q] = vs[(lc * kChunk + q) * BN + n];
            uint4 hw, lw;
            if constexpr (F16) {
                uint32_t h[4], l[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const __half2 hh = __floats2half2_rn(v[2 * q], v[2 * q + 1]);
                    const float2 hf = __half22float2(hh);
                    const __half2 ll = __floats2half2_rn(v[2 * q] - hf.x, v[2 * q + 1] - hf.y);
                    h[q] = half2_bits(hh);
                    l[q] = half2_bits(ll);
                }
                hw = make_uint4(h[0], h[1], h[2], h[3]);
                lw = make_uint4(l[0], l[1], l[2], l[3]);
            } else {
                uint32_t h[4], l[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    h[q] = __float_as_uint(v[q]);
                    l[q] = __float_as_uint(v[q] - __uint_as_float(h[q] & kTf32Mask));
                }
                hw = make_uint4(h[0], h[1], h[2], h[3]);
                lw = make_uint4(l[0], l[1], l[2], l[3]);
            }
            *reinterpret_cast<uint4*>(base + (int64_t)n * kRow + cp * 16) = hw;
            *reinterpret_cast<uint4*>(base + (int64_t)(BN + n) * kRow + cp * 16) = lw;
        }
        __syncthreads();
    }
}

// Mode-n product on the tensor cores: M^T (N x J, row-major) from M (J x N), the
// inner table of the "2-way MTTKRP" the product is computed as, and a row of
// J ones for its G table.
__global__ void ttm_prep_kernel(const float* __restrict__ M, int64_t J, int64_t N, float* __restrict__ mt,
                                float* __restrict__ ones) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < J * N; e += stride) {
        const int64_t j = e / N, i = e - j * N;
        mt[i * J + j] = M[e];
    }
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < J; e += stride) ones[e] = 1.f;
}

// ---------------------------------------------------------------------------
// Peak probe of the tensor pipe (measurement only).  One CTA per SM (the
// dynamic shared memory keeps a second one off); one thread issues `iters`
// M128 x N256 MMAs back to back -- kind::tf32 with K = 8, or kind::f16 with
// K = 16 -- from zero-filled shared-memory operands (64-byte swizzled K-major
// tiles) into one TMEM accumulator, then commits and waits (bounded).
// flops per MMA: 2 x 128 x 256 x K.
// ---------------------------------------------------------------------------
constexpr uint32_t kProbeSmem = 120 * 1024;

template <bool F16>
__global__ void __launch_bounds__(128, 1) mma_probe_kernel(int iters, uint32_t* status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~(uintptr_t)1023);
    constexpr uint32_t kA = 128 * 64, kB = 256 * 64;   // 64-byte rows
    uint64_t* done = reinterpret_cast<uint64_t*>(smem + kA + kB);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
    const int tid = threadIdx.x;
    for (uint32_t o = 16u * tid; o < kA + kB; o += 16u * blockDim.x)
        *reinterpret_cast<uint4*>(smem + o) = make_uint4(0u, 0u, 0u, 0u);
    if (tid == 0) {
        mbar_init(done, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (tid < 32) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(256));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    fence_proxy_async();   // the zero fill, seen by the tensor core's reads
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if (tid == 0) {
        const uint32_t a = sdesc_lo(smem_u32(smem)), b = sdesc_lo(smem_u32(smem + kA));
        if constexpr (F16) {
            const uint32_t idesc = (1u << 4) | ((uint32_t)(256 >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
            for (int i = 0; i < iters; ++i)
                asm volatile(
                    "{\n\t.reg .pred p;\n\t.reg .b64 da, db;\n\t"
                    "mov.b64 da, {%1, %3};\n\t"
                    "mov.b64 db, {%2, %3};\n\t"
                    "setp.ne.b32 p, %5, 0;\n\t"
                    "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %4, p;\n\t}\n" ::"r"(tmem),
                    "r"(a), "r"(b), "r"((uint32_t)(kDescSw64Hi >> 32)), "r"(idesc), "r"(i > 0 ? 1u : 0u));
        } else {
            const uint32_t idesc = (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(256 >> 3) << 17) |
                                   ((uint32_t)(128 >> 4) << 24);
            for (int i = 0; i < iters; ++i) mma_tf32_w(tmem, a, b, idesc, i > 0 ? 1u : 0u);
        }
        mma_commit(done);
        wait_drain(done, 0, status);
    }
    tc_fence_before();
    __syncthreads();
    if (tid < 32) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(256));
    }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

int g_sm_count = 0;

// test hook: launches left that withhold their first accumulator-ready signal
std::atomic<int> g_withhold_signal{0};

int sm_count() {
    if (g_sm_count == 0) {
        int dev = 0, n = 0;
        if (cudaGetDevice(&dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0)
            g_sm_count = n;
        else
            g_sm_count = 152;
        cudaGetLastError();  // a failed query on a host without a GPU leaves no sticky error
    }
    return g_sm_count;
}

int64_t cdiv64(int64_t a, int64_t b) { return (a + b - 1) / b; }

struct MapGeom {
    int rank;
    int slot[kRoles];
    uint64_t dim[5];
    uint64_t stride_el[5];  // element strides; stride_el[0] = 1
    uint32_t box[5];
};

// Tensor-map geometry of Y (elements of esize bytes: 4 for Y itself, 2 for its
// fp16 images) for mode plan mp; false if TMA cannot express it.
bool y_map_geom(const ModePlan& mp, const int64_t* dims, const int64_t* strides, int d, MapGeom& mg,
                int esize) {
    const ModeGeom& g = mp.g;
    const int k = g.k;
    struct Dim {
        int role;
        int64_t size, stride;
    } dl[kRoles];
    int n = 0;
    // pre modes split into the run before k and the run after k
    int64_t sizeP = 1, strideP = 0, sizeQ = 1, strideQ = 0;
    for (int t = 0; t < g.npm; ++t) {
        const int m = g.pm[t];
        if (m < k) {
            sizeP *= dims[m];
            strideP = strides[m];  // last (innermost) mode of the run
        } else {
            sizeQ *= dims[m];
            strideQ = strides[m];
        }
    }
    // the runs must be contiguous in memory (adjacent modes)
    for (int t = 0; t + 1 < g.npm; ++t) {
        const int m = g.pm[t], m2 = g.pm[t + 1];
        if ((m < k) == (m2 < k) && m2 != m + 1) return false;
    }
    (void)d;
    if (mp.tc_inner) {
        dl[n++] = {kRoleJq, g.J, g.IQ};   // j (stride I) — carried in the Jq role
        dl[n++] = {kRoleI, g.I, 1};
    } else {
        dl[n++] = {kRoleJq, g.Jq, 1};
        dl[n++] = {kRoleI, g.I, g.s_k};
        if (g.J > g.Jq) dl[n++] = {kRoleJp, g.J / g.Jq, g.IQ};
    }
    if (sizeP > 1) dl[n++] = {kRolePP, sizeP, strideP};
    if (sizeQ > 1) dl[n++] = {kRolePQ, sizeQ, strideQ};
    // the innermost (stride-1) dimension first, the others by increasing stride;
    // the small-I variant keeps (j, i, batch) as the first three dimensions so
    // that the tile rows come out as slot * I + i
    int first = -1;
    for (int t = 0; t < n; ++t)
        if (dl[t].stride == 1) first = t;
    if (first < 0) return false;
    Dim tmp = dl[0];
    dl[0] = dl[first];
    dl[first] = tmp;
    int fixed = 1;
    if (mp.tc_small) {
        const int batch_role = sizeQ > 1 ? kRolePQ : kRolePP;
        // K-major: (j, i, batch); innermost mode: (i, j, batch)
        const int second = mp.tc_inner ? (int)kRoleJq : (int)kRoleI;
        for (int want : {second, batch_role}) {
            for (int t = fixed; t < n; ++t)
                if (dl[t].role == want) {
                    tmp = dl[fixed];
                    dl[fixed] = dl[t];
                    dl[t] = tmp;
                    ++fixed;
                    break;
                }
        }
        if (fixed != 3) return false;
    }
    for (int t = fixed; t < n; ++t)
        for (int u = t + 1; u < n; ++u)
            if (dl[u].stride < dl[t].stride) {
                tmp = dl[t];
                dl[t] = dl[u];
                dl[u] = tmp;
            }
    if (n > 5) return false;
    mg.rank = n;
    for (int q = 0; q < kRoles; ++q) mg.slot[q] = -1;
    for (int t = 0; t < n; ++t) {
        mg.slot[dl[t].role] = t;
        mg.dim[t] = (uint64_t)dl[t].size;
        mg.stride_el[t] = (uint64_t)dl[t].stride;
        if (dl[t].size >= ((int64_t)1 << 31)) return false;
        if (t > 0 && ((dl[t].stride * esize) % 16 != 0 || dl[t].stride * esize >= ((int64_t)1 << 40)))
            return false;
        mg.box[t] = 1;
    }
    if (mp.tc_inner) {
        if (mg.slot[kRoleI] != 0) return false;   // i contiguous
        mg.box[mg.slot[kRoleJq]] = (uint32_t)(mp.tc_img_mn ? kBK4 : mp.tc_kw);
        if (mp.tc_small) {
            const int batch_role = sizeQ > 1 ? kRolePQ : kRolePP;
            if (mg.slot[batch_role] < 0 || mp.tc_ps < 2 || mp.tc_ps > 256 || (g.I * 4) % 16 != 0)
                return false;
            mg.box[0] = (uint32_t)g.I;
            mg.box[mg.slot[batch_role]] = (uint32_t)mp.tc_ps;
        } else {
            mg.box[0] = mp.tc_img_mn ? 64u : (uint32_t)kBM;   // MN-major: two boxes of 64 rows
        }
    } else {
        if (mg.slot[kRoleJq] != 0) return false;
        mg.box[0] = (uint32_t)mp.tc_kw;
        if (mp.tc_small) {
            // tc_ps consecutive pre indices along the fastest pre dimension
            const int batch_role = sizeQ > 1 ? kRolePQ : kRolePP;
            if (mg.slot[batch_role] < 0 || mp.tc_ps < 2 || mp.tc_ps > 256) return false;
            mg.box[mg.slot[kRoleI]] = (uint32_t)g.I;
            mg.box[mg.slot[batch_role]] = (uint32_t)mp.tc_ps;
        } else {
            mg.box[mg.slot[kRoleI]] = kBM;
        }
    }
    return true;
}

// Tensor-map geometry of the transposed images for the innermost mode: element
// (i, pi, j) at i * P + pi * J + j (P = npre * J); roles j (Jq, box 64), i (box
// 128) and pi (PP); false if TMA cannot express it.
bool timg_map_geom(const ModePlan& mp, MapGeom& mg) {
    const ModeGeom& g = mp.g;
    const int64_t P = g.npre * g.J;
    if ((g.J * 2) % 16 != 0 || (P * 2) % 16 != 0 || P * 2 >= ((int64_t)1 << 40)) return false;
    if (g.J >= ((int64_t)1 << 31) || g.I >= ((int64_t)1 << 31) || g.npre >= ((int64_t)1 << 31)) return false;
    mg.rank = 3;
    for (int q = 0; q < kRoles; ++q) mg.slot[q] = -1;
    mg.slot[kRoleJq] = 0;
    mg.slot[kRoleI] = 1;
    mg.slot[kRolePP] = 2;
    mg.dim[0] = (uint64_t)g.J;
    mg.dim[1] = (uint64_t)g.I;
    mg.dim[2] = (uint64_t)g.npre;
    mg.stride_el[0] = 1;
    mg.stride_el[1] = (uint64_t)P;
    mg.stride_el[2] = (uint64_t)g.J;
    mg.box[0] = (uint32_t)kBK4;
    mg.box[1] = kBM;
    mg.box[2] = 1;
    if (mp.tc_small) {
        // ps consecutive pre indices, all I_k rows: tile rows slot * I_k + i
        if (mp.tc_ps < 2 || mp.tc_ps > 256) return false;
        mg.box[1] = (uint32_t)g.I;
        mg.box[2] = (uint32_t)mp.tc_ps;
    }
    return true;
}

// The innermost mode can read transposed images when its inner group is the run
// of modes just before it and the pre modes are the modes before that (then
// (pi, j) is contiguous in the transposed layout).
bool timg_eligible(const ModeGeom& g, int d) {
    if (g.k != d - 1 || g.ngroup < 1) return false;
    for (int t = 0; t < g.ngroup; ++t)
        if (g.group[t] != d - 1 - g.ngroup + t) return false;
    for (int t = 0; t < g.npm; ++t)
        if (g.pm[t] != t) return false;
    return g.npm + g.ngroup == d - 1;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (fn == nullptr) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

template <bool INNER>
cudaError_t launch_h2(const TcArgs& args, dim3 grid, cudaStream_t s) {
    static bool attr_set[64] = {false};
    int dev = 0;
    cudaError_t e0 = cudaGetDevice(&dev);
    if (e0 != cudaSuccess) return e0;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        {
            // setmaxnreg.inc waits until the pool allotted at launch can serve it:
            // refuse a build whose launch allotment is below what the split assumes
            cudaFuncAttributes fa;
            cudaError_t e = cudaFuncGetAttributes(&fa, tc_h2_kernel<INNER>);
            if (e != cudaSuccess) return e;
            if (fa.numRegs < kH2RegsLaunch || fa.numRegs * kH2Threads > 65536) return cudaErrorInvalidConfiguration;
        }
        cudaError_t e = cudaFuncSetAttribute(tc_h2_kernel<INNER>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)SmemH2::kTotal);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    tc_h2_kernel<INNER><<<grid, kH2Threads, SmemH2::kTotal, s>>>(args);
    return cudaGetLastError();
}

template <int BN, bool SMALL = false, bool MN = false, bool CVT = false>
cudaError_t launch_img(const TcArgs& args, dim3 grid, cudaStream_t s) {
    static bool attr_set[64] = {false};
    int dev = 0;
    cudaError_t e0 = cudaGetDevice(&dev);
    if (e0 != cudaSuccess) return e0;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        // setmaxnreg.inc waits until the pool allotted at launch can serve it:
        // refuse a build whose launch allotment is below what the split assumes
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, tc_img_kernel<BN, SMALL, MN, CVT>);
        if (e != cudaSuccess) return e;
        const int need = CVT ? kCvtRegsLaunch : kImgRegsLaunch, threads = CVT ? kCvtThreads : kImgThreads;
        if (fa.numRegs < need || fa.numRegs * threads > 65536) return cudaErrorInvalidConfiguration;
        e = cudaFuncSetAttribute(tc_img_kernel<BN, SMALL, MN, CVT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)SmemImg<BN, SMALL>::kTotal);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    tc_img_kernel<BN, SMALL, MN, CVT><<<grid, CVT ? kCvtThreads : kImgThreads, SmemImg<BN, SMALL>::kTotal, s>>>(args);
    return cudaGetLastError();
}

template <bool INNER>
cudaError_t launch_tmem(const TcArgs& args, dim3 grid, cudaStream_t s) {
    static bool attr_set[64] = {false};
    int dev = 0;
    cudaError_t e0 = cudaGetDevice(&dev);
    if (e0 != cudaSuccess) return e0;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(tc_tmem_kernel<INNER>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)SmemT::kTotal);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    tc_tmem_kernel<INNER><<<grid, kTThreads, SmemT::kTotal, s>>>(args);
    return cudaGetLastError();
}

template <int BN, bool INNER, bool SMALL = false>
cudaError_t launch_main(const TcArgs& args, dim3 grid, cudaStream_t s) {
    using L = Smem<BN, INNER, SMALL>;
    static bool attr_set[64] = {false};
    int dev = 0;
    cudaError_t e0 = cudaGetDevice(&dev);
    if (e0 != cudaSuccess) return e0;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(tc_mttkrp_kernel<BN, INNER, SMALL>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::kTotal);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    tc_mttkrp_kernel<BN, INNER, SMALL><<<grid, Roles<INNER>::kThreads, L::kTotal, s>>>(args);
    return cudaGetLastError();
}

size_t bimg_bytes(const ModePlan& mp) {
    // per K-step: hi and lo images of bn rows x tc_kw elements (64-byte rows of
    // 16 fp32 or 32 fp16; 128-byte rows of 64 fp16 for tc_img)
    const size_t row = mp.tc_img ? 128 : 64;
    return (size_t)cdiv64(mp.g.R, mp.bn) * mp.tc_ks * 2 * (size_t)mp.bn * row;
}

// fp16 split: the column scales follow the images
size_t colscale_offset(const ModePlan& mp) { return (bimg_bytes(mp) + 255) / 256 * 256; }

// Small I_k (16..64): floor(128 / I_k) pre indices are stacked in one 128-row
// tile (for the innermost mode the TMA box's i extent, I_k * 4 bytes, must be a
// multiple of 16).
bool small_eligible(const ModeGeom& g) {
    return g.I >= 16 && g.I <= 64 && g.npre >= 2 && (g.s_k != 1 || g.I % 4 == 0);
}

}  // namespace

size_t tc_binner_bytes(const ModePlan& mp) {
    return (mp.tc_h2 || mp.tc_img) ? colscale_offset(mp) + (size_t)mp.g.R * sizeof(float) : bimg_bytes(mp);
}

bool tc_prefer(const ModePlan& mp) {
    // the 128-row tile must be reasonably full (directly, or with several pre
    // indices stacked in it for small I_k) and the rank large enough for the
    // tensor-core products to pay off
    return mp.g.R >= 32 && (mp.g.I >= 96 || small_eligible(mp.g));
}

bool tc_plan(const Plan& p, ModePlan& mp, bool allow_fp16) {
    const ModeGeom& g = mp.g;
    mp.path = MTTKRP_PATH_TC;
    mp.tc_inner = (g.s_k == 1) ? 1 : 0;
    mp.tc_small = small_eligible(g) ? 1 : 0;
    mp.tc_ps = mp.tc_small ? (int)(kBM / g.I) : 1;
    // innermost mode with large R: A staged in tensor memory (the i-contiguous
    // tile is transposed on the way into TMEM, no shared-memory round trip)
    mp.tc_tmem = (!mp.explicit_krp && !mp.tc_small && g.R >= kTmemMinR && mp.tc_inner) ? 1 : 0;
    // the two-term fp16 split in tensor memory (128 x 224 tiles) does a K-step
    // about 1.4 times faster than the tf32 kernel (128 x 256 tiles): it wins
    // unless its narrower tiles waste more columns than that
    {
        const int64_t h2_cols = cdiv64(g.R, kH2BN) * kH2BN * 10;
        const int64_t tf_cols = cdiv64(g.R, 256) * 256 * 14;
        mp.tc_h2 = (allow_fp16 && !mp.explicit_krp && !mp.tc_small && g.R >= kH2MinR && h2_cols < tf_cols) ? 1 : 0;
    }
    if (mp.tc_h2) mp.tc_tmem = 1;
    mp.tc_kw = mp.tc_h2 ? kBK2 : kBK;
    mp.bm = kBM;
    mp.bn = mp.tc_h2 ? kH2BN : mp.tc_tmem ? kTBN : g.R >= 192 ? 256 : (g.R > 64 ? 128 : 64);
    // K-major modes with a wide enough R: the fp16 split streamed from images of
    // Y written once per call (no producer warps, both operands in shared
    // memory, 128 x 256 or 128 x 128 tiles, K-steps of 64 indices); the q-block
    // length must not be padded to K-steps by much
    mp.tc_img = 0;
    mp.tc_img_t = 0;
    // the images take 4 bytes an element per layout (natural, transposed); above
    // 12 Gi elements (48 GiB of Y) they would crowd the tensor out of HBM, and
    // the kernels that convert Y per CTA take over
    int64_t numel = 1;
    for (int t = 0; t < p.d; ++t) numel *= p.dims[t];
    if (allow_fp16 && g.R >= kImgMinR && numel <= ((int64_t)12 << 30)) {
        ModePlan t = mp;
        t.tc_img = 1;
        t.tc_h2 = 0;
        t.tc_tmem = 0;
        t.tc_kw = kBK4;
        // 128 x 64 tiles for small R; else 256 or 128 columns, whichever wastes
        // fewer (256 preferred within 15 %)
        t.bn = g.R <= 64 ? 64 : (cdiv64(g.R, 256) * 256 * 20 <= cdiv64(g.R, 128) * 128 * 23 ? 256 : 128);
        if (mp.tc_small && t.bn > 128) t.bn = 128;   // per-row G loads: 128-column tiles at most
        MapGeom mgi;
        if (!mp.tc_inner) {
            if (cdiv64(g.Jq, kBK4) * kBK4 * 8 <= g.Jq * 9 && y_map_geom(t, p.dims, p.strides, p.d, mgi, 2)) mp = t;
        } else if (!mp.tc_small && cdiv64(g.J, kBK4) * kBK4 * 8 <= g.J * 9 &&
                   (t.tc_img_mn = 1, y_map_geom(t, p.dims, p.strides, p.d, mgi, 2))) {
            // the innermost mode from the natural images, A MN-major (boxes of
            // 64 i x 64 j; the i stride of the image a 16-byte multiple)
            mp = t;
        } else if (timg_eligible(g, p.d) && cdiv64(g.J, kBK4) * kBK4 * 8 <= g.J * 9) {
            t.tc_img_mn = 0;
            // the innermost mode from the transposed images (written in the same
            // pass as the others); the K-steps run over j alone
            t.tc_img_t = 1;
            if (timg_map_geom(t, mgi)) mp = t;
        }
    }
    if (mp.tc_inner) {
        if (g.J > g.Jq && g.Jq != 1) return false;
        mp.tc_jq_steps = 1;
        mp.tc_ks = (int)cdiv64(g.J, mp.tc_kw);
    } else {
        mp.tc_jq_steps = (int)cdiv64(g.Jq, mp.tc_kw);
        mp.tc_ks = (int)((g.J / g.Jq) * mp.tc_jq_steps);
    }
    if (mp.tc_img_t || mp.tc_img_mn) mp.tc_jq_steps = mp.tc_ks;   // the j role carries the whole K-step offset
    if ((!mp.tc_small && cdiv64(g.I, kBM) > 65535) || g.npre >= ((int64_t)1 << 31)) return false;
    MapGeom mg;
    if (mp.tc_img_t ? !timg_map_geom(mp, mg) : !y_map_geom(mp, p.dims, p.strides, p.d, mg, mp.tc_img ? 2 : 4))
        return false;
    // split count: fill whole waves of one CTA per SM, at least two drain
    // chunks per CTA where possible
    const int64_t tiles = (mp.tc_small ? 1 : cdiv64(g.I, kBM)) * cdiv64(g.R, mp.bn);
    const int64_t sms = sm_count();
    if (mp.explicit_krp) {
        // one pre index: split the B chunks instead
        if (cdiv64(g.R, mp.bn) > kKrpMaxBN || mp.bn > kKrpMaxBN) return false;
        const int ck = mp.tc_img ? kImgCK
                                 : (int)(((mp.tc_inner ? kBResInnerKB : kBResKB) * 1024) /
                                         (2 * mp.bn * kBK * 4));
        const int64_t njc = cdiv64(mp.tc_ks, ck);
        int64_t best = 1;
        double best_eff = -1.0;
        for (int64_t S = 1; S <= njc && S * tiles <= 8 * sms; ++S) {
            const int64_t ctas = S * tiles;
            const double eff = (double)ctas / (double)(cdiv64(ctas, sms) * sms);
            if (eff > best_eff + 0.02) {
                best_eff = eff;
                best = S;
            }
        }
        const int64_t jcps = cdiv64(njc, best);
        mp.jc_per_split = (int)jcps;
        mp.splits = cdiv64(njc, jcps);
        mp.pre_per_split = 1;
        return true;
    }
    const int64_t smax = g.npre;
    int64_t best = 1;
    double best_eff = -1.0;
    for (int64_t S = 1; S <= smax && S * tiles <= 8 * sms; ++S) {
        const int64_t ctas = S * tiles;
        const double eff = (double)ctas / (double)(cdiv64(ctas, sms) * sms);
        if (eff > best_eff + 0.02) {
            best_eff = eff;
            best = S;
        }
    }
    mp.pre_per_split = cdiv64(g.npre, best);
    mp.splits = cdiv64(g.npre, mp.pre_per_split);
    return true;
}

int tc_prepare(const Plan& p, const ModePlan& mp, const float* Y, void* ws, cudaStream_t stream, int* nlaunch,
               char* errbuf, size_t errlen) {
    *nlaunch = 0;
    if (!(mp.tc_h2 || mp.tc_img)) return MTTKRP_OK;
    if ((reinterpret_cast<uintptr_t>(Y) & 15) != 0) {
        snprintf(errbuf, errlen, "tensor-core path needs a 16-byte aligned Y");
        return MTTKRP_ERR_INVALID;
    }
    uint8_t* ws_base = static_cast<uint8_t*>(ws);
    uint32_t* ymax = reinterpret_cast<uint32_t*>(ws_base);   // reserved first bytes
    uint32_t* slab = reinterpret_cast<uint32_t*>(ws_base + p.off_slab);
    int64_t numel = 1;
    for (int t = 0; t < p.d; ++t) numel *= p.dims[t];
    const int64_t slab_len = numel / p.nslab;
    cudaError_t e = cudaSuccess;
    // The maxima of a call that also writes the images (the common case) are
    // sampled; the image pass checks every scaled value and, if one left the
    // fp16 range, a second max pass (over all of Y, on top of the samples) and
    // a second image pass run; otherwise those two launches return at once.
    // Plans whose first fp16 mode converts per CTA take the exact maxima.
    uint32_t* ovf = slab + p.nslab;   // the image pass's out-of-range flag
    const bool sampled = !p.ymax_ready && mp.tc_img && !p.img_ready;
    // the mode's own main kernel can write the images while it converts its
    // tiles (then it sets the flag, and the gated redo launches follow it)
    const bool fuse = sampled && mp.g.k == p.fuse_mode && tc_fuse_eligible(p, mp);
    int64_t max_blocks = cdiv64(cdiv64(slab_len, kSlabUnit) * p.nslab, 4);
    if (max_blocks > 152 * 8) max_blocks = 152 * 8;
    if (!p.ymax_ready) {
        // largest magnitude of every slab of mode 0 and of the whole tensor
        e = cudaMemsetAsync(ymax, 0, sizeof(uint32_t), stream);
        if (e == cudaSuccess) e = cudaMemsetAsync(slab, 0, (size_t)(p.nslab + 1) * sizeof(uint32_t), stream);
        if (e == cudaSuccess) {
            if (sampled) {
                const int64_t nch = cdiv64(slab_len, kSampleChunk);
                const int64_t per = cdiv64(nch, nch > kSampleEvery ? kSampleEvery : 1);
                int64_t blocks = cdiv64(per * p.nslab, 8);
                if (blocks > 152 * 8) blocks = 152 * 8;
                slabsample_kernel<<<(unsigned)blocks, 256, 0, stream>>>(Y, p.nslab, slab_len, slab, ymax);
            } else {
                slabmax_kernel<<<(unsigned)max_blocks, 256, 0, stream>>>(Y, p.nslab, slab_len, slab, ymax, nullptr);
            }
            e = cudaGetLastError();
        }
        if (e == cudaSuccess) {
            p.ymax_ready = 1;
            ++*nlaunch;
        }
    }
    if (e == cudaSuccess && mp.tc_img && !p.img_ready && fuse) {
        p.img_ready = 1;
        p.fuse_pending = 1;
    } else if (e == cudaSuccess && mp.tc_img && !p.img_ready) {
        // every image the plan's tc_img modes read, in one pass over Y
        const size_t img_half = ((size_t)numel * 2 + 255) / 256 * 256;
        __half* img_hi = reinterpret_cast<__half*>(ws_base + mp.off_img);
        __half* img_lo = reinterpret_cast<__half*>(ws_base + mp.off_img + img_half);
        __half* timg_hi = reinterpret_cast<__half*>(ws_base + mp.off_timg);
        __half* timg_lo = reinterpret_cast<__half*>(ws_base + mp.off_timg + img_half);
        // pass 0: with the maxima as they are, flagging out-of-range values when
        // they were sampled; pass 1 (sampled maxima only): the exact redo, which
        // runs only if the flag is set
        for (int pass = 0; pass < (sampled ? 2 : 1) && e == cudaSuccess; ++pass) {
            uint32_t* flag_out = (sampled && pass == 0) ? ovf : nullptr;
            const uint32_t* enable = pass == 1 ? ovf : nullptr;
            if (pass == 1) {
                slabmax_kernel<<<(unsigned)max_blocks, 256, 0, stream>>>(Y, p.nslab, slab_len, slab, ymax, enable);
                if ((e = cudaGetLastError()) != cudaSuccess) break;
                ++*nlaunch;
            }
            if (p.img_t) {
                const int64_t In = p.dims[p.d - 1];
                const int64_t P = numel / In;
                int64_t blocks = cdiv64(P, 64) * cdiv64(In, 128);
                if (blocks > 152 * 16) blocks = 152 * 16;
                // (I_{d-1} < 64: whole rows per tile, read flat; the 16-byte
                // alignment of every tile start holds because tiles are 64 rows)
                const int64_t rps = P / p.nslab;
                if (In % 4 == 0)
                    split_image_t_kernel<true><<<(unsigned)blocks, 256, 0, stream>>>(
                        Y, P, In, slab, ymax, rps, img_hi, img_lo, timg_hi, timg_lo, p.img_nat, flag_out, enable);
                else
                    split_image_t_kernel<false><<<(unsigned)blocks, 256, 0, stream>>>(
                        Y, P, In, slab, ymax, rps, img_hi, img_lo, timg_hi, timg_lo, p.img_nat, flag_out, enable);
            } else {
                split_image_kernel<<<(unsigned)max_blocks, 256, 0, stream>>>(Y, p.nslab, slab_len, slab, ymax,
                                                                            img_hi, img_lo, flag_out, enable);
            }
            e = cudaGetLastError();
            if (e == cudaSuccess) ++*nlaunch;
        }
        if (e == cudaSuccess) p.img_ready = 1;
    }
    if (e != cudaSuccess) {
        snprintf(errbuf, errlen, "fp16 split pass: %s", cudaGetErrorString(e));
        return MTTKRP_ERR_CUDA;
    }
    return MTTKRP_OK;
}

bool tc_fuse_eligible(const Plan& p, const ModePlan& mp) {
    if (mp.path != MTTKRP_PATH_TC || !mp.tc_img || mp.tc_img_mn || mp.tc_img_t || mp.tc_small || mp.explicit_krp ||
        p.img_t || !p.img_nat || mp.g.J != mp.g.Jq || mp.g.Jq % kBK4 != 0)
        return false;
    // one column tile: with several, each would convert the same Y tiles
    if (cdiv64(mp.g.R, mp.bn) != 1) return false;
    MapGeom mg;
    return y_map_geom(mp, p.dims, p.strides, p.d, mg, 4) && y_map_geom(mp, p.dims, p.strides, p.d, mg, 2);
}

int tc_pick_fuse_mode(const Plan& p) {
    int first = -1;
    for (int k = 0; k < p.d; ++k) {
        const ModePlan& mp = p.mode[k];
        if (!tc_fuse_eligible(p, mp)) continue;
        if (mp.g.s_k == mp.g.Jq) return k;   // 128 rows x Jq of one pre index: one contiguous block
        if (first < 0) first = k;
    }
    return first;
}

namespace {
// phase 0: the mode as planned; 1: the main kernel converts Y in place and
// writes the images (p.fuse_pending); 2: the exact redo of phase 1's main
// kernel, run only if its conversion flagged a value (the Binner scales and B
// images of phase 1 are still in place)
int tc_run_phase(const Plan& p, const ModePlan& mp, const float* Y, const float* const* factors,
                 const float* gtab, const int64_t* basetab, void* binner_ws, float* dst, cudaStream_t stream,
                 int* nlaunch, cudaEvent_t* start_ev, char* errbuf, size_t errlen, int phase) {
    (void)basetab;
    *nlaunch = 0;
    const ModeGeom& g = mp.g;
    if ((reinterpret_cast<uintptr_t>(Y) & 15) != 0) {
        snprintf(errbuf, errlen, "tensor-core path needs a 16-byte aligned Y");
        return MTTKRP_ERR_INVALID;
    }
    MapGeom mg;
    if (mp.tc_img_t ? !timg_map_geom(mp, mg) : !y_map_geom(mp, p.dims, p.strides, p.d, mg, mp.tc_img ? 2 : 4)) {
        snprintf(errbuf, errlen, "mode %d: Y view not expressible as a TMA tensor map", g.k);
        return MTTKRP_ERR_UNSUPPORTED;
    }
    PFN_cuTensorMapEncodeTiled_v12000 encode = encode_fn();
    if (encode == nullptr) {
        snprintf(errbuf, errlen, "cuTensorMapEncodeTiled entry point not available");
        return MTTKRP_ERR_CUDA;
    }
    TcArgs args;
    memset(&args, 0, sizeof(args));
    // fp16 images of Y (tc_img): hi then lo, in the region every tc_img mode shares
    uint8_t* ws_base = static_cast<uint8_t*>(binner_ws) - mp.off_binner;
    int64_t numel = 1;
    for (int t = 0; t < p.d; ++t) numel *= p.dims[t];
    const size_t img_half = ((size_t)numel * 2 + 255) / 256 * 256;
    __half* img_hi = reinterpret_cast<__half*>(ws_base + mp.off_img);
    __half* img_lo = reinterpret_cast<__half*>(ws_base + mp.off_img + img_half);
    __half* timg_hi = reinterpret_cast<__half*>(ws_base + mp.off_timg);
    __half* timg_lo = reinterpret_cast<__half*>(ws_base + mp.off_timg + img_half);
    __half* map_hi = mp.tc_img_t ? timg_hi : img_hi;
    __half* map_lo = mp.tc_img_t ? timg_lo : img_lo;
    const size_t esize = mp.tc_img ? 2 : 4;
    cuuint64_t gdim[5], gstride[4];
    cuuint32_t box[5], estr[5];
    for (int t = 0; t < mg.rank; ++t) {
        gdim[t] = mg.dim[t];
        box[t] = mg.box[t];
        estr[t] = 1;
        if (t > 0) gstride[t - 1] = mg.stride_el[t] * esize;
    }
    // L2 promotion: a copy's L2 fills are widened to 256 bytes, which prefetches
    // the next K-step of the same rows when rows and strides are 256-byte
    // multiples; with shorter or unaligned rows (e.g. 800-byte rows of 400
    // fp16) the widened fills straddle rows and the data is fetched about twice,
    // so the fill width follows the alignment of the row length and strides
    uint64_t align = (uint64_t)gdim[0] * esize;
    for (int t = 0; t + 1 < mg.rank; ++t) align |= (uint64_t)gstride[t];
    const CUtensorMapL2promotion promo = (align % 256 == 0)   ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B
                                         : (align % 128 == 0) ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B
                                         : (align % 64 == 0)  ? CU_TENSOR_MAP_L2_PROMOTION_L2_64B
                                                              : CU_TENSOR_MAP_L2_PROMOTION_NONE;
    CUresult cr;
    if (mp.tc_img) {
        // 64 fp16 = 128-byte rows, 128-byte swizzle (the MMA descriptors' layout)
        cr = encode(&args.ymap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, (cuuint32_t)mg.rank, map_hi, gdim, gstride,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, promo,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (cr == CUDA_SUCCESS)
            cr = encode(&args.ymap_lo, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, (cuuint32_t)mg.rank, map_lo, gdim,
                        gstride, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, promo,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
        cr = encode(&args.ymap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, (cuuint32_t)mg.rank, const_cast<float*>(Y),
                    gdim, gstride, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    mp.tc_inner ? CU_TENSOR_MAP_SWIZZLE_NONE
                    : mp.tc_h2  ? CU_TENSOR_MAP_SWIZZLE_128B   // 32 fp32 = 128-byte rows
                                : CU_TENSOR_MAP_SWIZZLE_64B,
                    promo, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    if (cr == CUDA_SUCCESS && phase == 1) {
        // fp32 Y in 32-index boxes (128-byte rows, the 128-byte swizzle)
        MapGeom mf;
        if (!y_map_geom(mp, p.dims, p.strides, p.d, mf, 4)) {
            snprintf(errbuf, errlen, "mode %d: Y view not expressible as an fp32 TMA tensor map", g.k);
            return MTTKRP_ERR_UNSUPPORTED;
        }
        cuuint64_t fdim[5], fstride[4];
        cuuint32_t fbox[5];
        for (int t = 0; t < mf.rank; ++t) {
            fdim[t] = mf.dim[t];
            fbox[t] = mf.box[t];
            if (t > 0) fstride[t - 1] = mf.stride_el[t] * 4;
        }
        fbox[0] = 32;
        uint64_t falign = (uint64_t)fdim[0] * 4;
        for (int t = 0; t + 1 < mf.rank; ++t) falign |= (uint64_t)fstride[t];
        const CUtensorMapL2promotion fpromo = (falign % 256 == 0)   ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B
                                              : (falign % 128 == 0) ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B
                                                                    : CU_TENSOR_MAP_L2_PROMOTION_NONE;
        cr = encode(&args.yfmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, (cuuint32_t)mf.rank, const_cast<float*>(Y), fdim,
                    fstride, fbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, fpromo,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    if (cr != CUDA_SUCCESS) {
        snprintf(errbuf, errlen, "cuTensorMapEncodeTiled failed (%d)", (int)cr);
        return MTTKRP_ERR_CUDA;
    }
    args.rank = mg.rank;
    for (int q = 0; q < kRoles; ++q) args.slot[q] = mg.slot[q];

    // B images
    float* bimg = static_cast<float*>(binner_ws);
    float* colscale = reinterpret_cast<float*>(static_cast<uint8_t*>(binner_ws) + colscale_offset(mp));
    // the first bytes of the workspace (reserved region) hold max |Y| as fp32 bits
    uint32_t* ymax = reinterpret_cast<uint32_t*>(ws_base);
    if ((mp.tc_h2 || mp.tc_img) && phase != 2) {
        ColScaleArgs c;
        memset(&c, 0, sizeof(c));
        c.ngroup = g.ngroup;
        for (int t = 0; t < g.ngroup; ++t) {
            c.gdim[t] = p.dims[g.group[t]];
            c.gfac[t] = factors[g.group[t]];
        }
        c.R = g.R;
        c.out = colscale;
        colscale_kernel<<<(unsigned)cdiv64(g.R, 32), 1024, 0, stream>>>(c);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) {
            snprintf(errbuf, errlen, "scale launch: %s", cudaGetErrorString(e));
            return MTTKRP_ERR_CUDA;
        }
        ++*nlaunch;
    }
    if (phase == 2) {
        // B images as phase 1 left them
    } else if (mp.explicit_krp) {
        KrpImgArgs b;
        memset(&b, 0, sizeof(b));
        const int last = g.group[g.ngroup - 1];
        b.t1 = reinterpret_cast<const float*>(ws_base + mp.off_t1);
        b.alast = factors[last];
        b.ilast = p.dims[last];
        b.colscale = colscale;
        b.R = g.R;
        b.J = g.J;
        b.Jq = g.Jq;
        b.BN = mp.bn;
        b.KS = mp.tc_ks;
        b.jq_steps = mp.tc_jq_steps;
        b.inner = mp.tc_inner;
        b.nblocks = cdiv64(g.R, mp.bn) * mp.tc_ks;
        b.out = bimg;
        int64_t blocks = b.nblocks < 152 * 8 ? b.nblocks : 152 * 8;
        const int kw = mp.tc_img ? kBK4 : kBK;
        const size_t smem = (size_t)kw * mp.bn * sizeof(float);
        cudaError_t e = cudaSuccess;
        if (mp.tc_img) {
            e = cudaFuncSetAttribute(krp_image_kernel<kBK4, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)(kBK4 * kKrpMaxBN * sizeof(float)));
            if (e == cudaSuccess) krp_image_kernel<kBK4, true><<<(unsigned)blocks, 256, smem, stream>>>(b);
        } else {
            krp_image_kernel<kBK, false><<<(unsigned)blocks, 256, smem, stream>>>(b);
        }
        if (e == cudaSuccess) e = cudaGetLastError();
        if (e != cudaSuccess) {
            snprintf(errbuf, errlen, "Khatri-Rao image launch: %s", cudaGetErrorString(e));
            return MTTKRP_ERR_CUDA;
        }
        ++*nlaunch;
    } else {
        BImgArgs b;
        memset(&b, 0, sizeof(b));
        b.ngroup = g.ngroup;
        for (int t = 0; t < g.ngroup; ++t) {
            b.gdim[t] = p.dims[g.group[t]];
            b.gfac[t] = factors[g.group[t]];
        }
        b.R = g.R;
        b.J = g.J;
        b.Jq = g.Jq;
        b.BN = mp.bn;
        b.KS = mp.tc_ks;
        b.jq_steps = mp.tc_jq_steps;
        b.inner = mp.tc_inner;
        b.nblocks = cdiv64(g.R, mp.bn) * mp.tc_ks;
        b.out = bimg;
        const int64_t n = b.nblocks * 2 * mp.bn * mp.tc_kw;
        int64_t blocks = cdiv64(n, 256);
        if (blocks > 152 * 16) blocks = 152 * 16;
        cudaError_t e;
        if (mp.tc_img) {
            e = launch_bimage_f16<kBK4>(b, colscale, stream);
        } else if (mp.tc_h2) {
            e = launch_bimage_f16<kBK2>(b, colscale, stream);
        } else {
            tc_bimage_kernel<<<(unsigned)blocks, 256, 0, stream>>>(b);
            e = cudaGetLastError();
        }
        if (e != cudaSuccess) {
            snprintf(errbuf, errlen, "B image launch: %s", cudaGetErrorString(e));
            return MTTKRP_ERR_CUDA;
        }
        ++*nlaunch;
    }

    // the pre index pi = (p-side, q-side) in C order
    int64_t nQ = 1;
    for (int t = 0; t < g.npm; ++t)
        if (g.pm[t] > g.k) nQ *= p.dims[g.pm[t]];
    if (mp.tc_img_t) nQ = 1;   // one pre dimension in the transposed layout
    args.bimg = bimg;
    args.gtab = gtab;
    args.dst = dst;
    args.dst_split_stride = g.I * g.R;
    args.I = g.I;
    args.R = g.R;
    args.npre = g.npre;
    args.pre_per_split = mp.pre_per_split;
    args.nQ = nQ;
    args.KS = mp.tc_ks;
    args.jq_steps = mp.tc_jq_steps;
    args.ps = mp.tc_small ? mp.tc_ps : 1;
    args.jc_per_split = mp.explicit_krp ? mp.jc_per_split : 0;
    args.batch_len = nQ > 1 ? nQ : g.npre;
    args.y_box_bytes = mp.tc_img ? (uint32_t)kBK4 * 2u *   // one fp16 image tile
                                       (mp.tc_small ? (uint32_t)(g.I * mp.tc_ps) : (uint32_t)kBM)
                                 : (uint32_t)mp.tc_kw * 4u * (mp.tc_small ? (uint32_t)(g.I * mp.tc_ps) : (uint32_t)kBM);
    args.ymax_bits = ymax;
    args.slab_bits = reinterpret_cast<const uint32_t*>(ws_base + p.off_slab);
    args.slab_rows = (p.slab_on && g.k == 0) ? 1 : 0;
    args.slab_div = (p.slab_on && g.k != 0) ? g.npre / p.nslab : g.npre;
    args.colscale = colscale;
    {
        int n = g_withhold_signal.load();
        while (n > 0 && !g_withhold_signal.compare_exchange_weak(n, n - 1)) {
        }
        args.withhold_signal = n > 0 ? 1 : 0;
    }
    args.status = tc_status_ptr();
    if (args.status == nullptr) {
        snprintf(errbuf, errlen, "device status word unavailable");
        return MTTKRP_ERR_CUDA;
    }
    uint32_t* ovf = reinterpret_cast<uint32_t*>(ws_base + p.off_slab) + p.nslab;
    if (phase == 1) args.ovf = ovf;
    if (phase == 2) args.enable = ovf;
    if (start_ev) cudaEventRecord(*start_ev, stream);
    dim3 grid((unsigned)cdiv64(g.R, mp.bn), mp.tc_small ? 1u : (unsigned)cdiv64(g.I, kBM),
              (unsigned)mp.splits);
    cudaError_t e;
    if (phase == 1) {
        e = mp.bn == 256 ? launch_img<256, false, false, true>(args, grid, stream)
          : mp.bn == 128 ? launch_img<128, false, false, true>(args, grid, stream)
                         : launch_img<64, false, false, true>(args, grid, stream);
    } else if (mp.tc_img) {
        if (mp.tc_small)
            e = mp.bn == 128 ? launch_img<128, true>(args, grid, stream) : launch_img<64, true>(args, grid, stream);
        else
            e = mp.tc_img_mn ? (mp.bn == 256 ? launch_img<256, false, true>(args, grid, stream)
                                : mp.bn == 128 ? launch_img<128, false, true>(args, grid, stream)
                                               : launch_img<64, false, true>(args, grid, stream))
                             : (mp.bn == 256 ? launch_img<256>(args, grid, stream)
                                : mp.bn == 128 ? launch_img<128>(args, grid, stream)
                                               : launch_img<64>(args, grid, stream));
    } else if (mp.tc_h2) {
        e = mp.tc_inner ? launch_h2<true>(args, grid, stream) : launch_h2<false>(args, grid, stream);
    } else if (mp.tc_tmem) {
        e = mp.tc_inner ? launch_tmem<true>(args, grid, stream) : launch_tmem<false>(args, grid, stream);
    } else if (mp.tc_small && mp.tc_inner) {
        e = mp.bn == 256 ? launch_main<256, true, true>(args, grid, stream)
          : mp.bn == 128 ? launch_main<128, true, true>(args, grid, stream)
                         : launch_main<64, true, true>(args, grid, stream);
    } else if (mp.tc_small) {
        e = mp.bn == 256 ? launch_main<256, false, true>(args, grid, stream)
          : mp.bn == 128 ? launch_main<128, false, true>(args, grid, stream)
                         : launch_main<64, false, true>(args, grid, stream);
    } else if (mp.tc_inner) {
        e = mp.bn == 256 ? launch_main<256, true>(args, grid, stream)
          : mp.bn == 128 ? launch_main<128, true>(args, grid, stream)
                         : launch_main<64, true>(args, grid, stream);
    } else {
        e = mp.bn == 256 ? launch_main<256, false>(args, grid, stream)
          : mp.bn == 128 ? launch_main<128, false>(args, grid, stream)
                         : launch_main<64, false>(args, grid, stream);
    }
    if (e != cudaSuccess) {
        snprintf(errbuf, errlen, "tensor-core kernel launch: %s", cudaGetErrorString(e));
        return MTTKRP_ERR_CUDA;
    }
    ++*nlaunch;
    return MTTKRP_OK;
}
}  // namespace

int tc_run(const Plan& p, const ModePlan& mp, const float* Y, const float* const* factors,
           const float* gtab, const int64_t* basetab, void* binner_ws, float* dst,
           cudaStream_t stream, int* nlaunch, cudaEvent_t* start_ev, char* errbuf, size_t errlen) {
    return tc_run_phase(p, mp, Y, factors, gtab, basetab, binner_ws, dst, stream, nlaunch, start_ev, errbuf, errlen,
                        p.fuse_pending ? 1 : 0);
}

const uint32_t* tc_redo_flag(const Plan& p, void* ws) {
    return reinterpret_cast<const uint32_t*>(static_cast<uint8_t*>(ws) + p.off_slab) + p.nslab;
}

int tc_redo_images(const Plan& p, const ModePlan& mp, const float* Y, void* ws, cudaStream_t stream, int* nlaunch,
                   char* errbuf, size_t errlen) {
    *nlaunch = 0;
    uint8_t* ws_base = static_cast<uint8_t*>(ws);
    uint32_t* ymax = reinterpret_cast<uint32_t*>(ws_base);
    uint32_t* slab = reinterpret_cast<uint32_t*>(ws_base + p.off_slab);
    const uint32_t* ovf = tc_redo_flag(p, ws);
    int64_t numel = 1;
    for (int t = 0; t < p.d; ++t) numel *= p.dims[t];
    const int64_t slab_len = numel / p.nslab;
    const size_t img_half = ((size_t)numel * 2 + 255) / 256 * 256;
    __half* img_hi = reinterpret_cast<__half*>(ws_base + mp.off_img);
    __half* img_lo = reinterpret_cast<__half*>(ws_base + mp.off_img + img_half);
    int64_t blocks = cdiv64(cdiv64(slab_len, kSlabUnit) * p.nslab, 4);
    if (blocks > 152 * 8) blocks = 152 * 8;
    slabmax_kernel<<<(unsigned)blocks, 256, 0, stream>>>(Y, p.nslab, slab_len, slab, ymax, ovf);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) {
        split_image_kernel<<<(unsigned)blocks, 256, 0, stream>>>(Y, p.nslab, slab_len, slab, ymax, img_hi, img_lo,
                                                                 nullptr, ovf);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) {
        snprintf(errbuf, errlen, "fp16 split redo: %s", cudaGetErrorString(e));
        return MTTKRP_ERR_CUDA;
    }
    *nlaunch = 2;
    return MTTKRP_OK;
}

int tc_redo_main(const Plan& p, const ModePlan& mp, const float* Y, const float* const* factors,
                 const float* gtab, const int64_t* basetab, void* binner_ws, float* dst,
                 cudaStream_t stream, int* nlaunch, char* errbuf, size_t errlen) {
    p.fuse_pending = 0;
    return tc_run_phase(p, mp, Y, factors, gtab, basetab, binner_ws, dst, stream, nlaunch, nullptr, errbuf, errlen,
                        2);
}

cudaError_t tc_launch_mma_probe(int kind, int blocks, int iters, cudaStream_t s) {
    static bool attr_set[64][2] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    uint32_t* status = tc_status_ptr();
    if (status == nullptr) return cudaErrorInvalidSymbol;
    const int f16 = kind == 1 ? 1 : 0;
    if (!attr_set[dev][f16]) {
        e = f16 ? cudaFuncSetAttribute(mma_probe_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kProbeSmem)
                : cudaFuncSetAttribute(mma_probe_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kProbeSmem);
        if (e != cudaSuccess) return e;
        attr_set[dev][f16] = true;
    }
    if (f16)
        mma_probe_kernel<true><<<blocks, 128, kProbeSmem, s>>>(iters, status);
    else
        mma_probe_kernel<false><<<blocks, 128, kProbeSmem, s>>>(iters, status);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Mode-n product T = X x_n M on the tensor cores.  With X viewed [P, N, Q] and T
// [P, J, Q], T[p, j, q] = sum_i X[p, i, q] M[j, i] is the mode-0 MTTKRP of the
// two-way array Z[(p, q), i] with the single factor M^T (rank J): rows (p, q),
// contraction over i, columns j, G a row of ones.  Z is read from the natural
// fp16 images of X: K-major when Q = 1 (the innermost mode), else MN-major (q
// contiguous, two 64-row halves of one p each, so Q must be a multiple of 64).
// One scale for the whole of X (a single slab).
// ---------------------------------------------------------------------------
namespace {
struct TtmLayout {
    int bn, ks;
    int64_t rows;
    size_t off_mt, off_ones, off_bimg, off_colscale, off_img, total;
};

bool ttm_layout(int64_t P, int64_t N, int64_t Q, int64_t J, TtmLayout& l) {
    const int64_t numel = P * N * Q;
    l.rows = Q == 1 ? P : P * Q;
    if (J < kImgMinR || J > 65536 || N < 16 || cdiv64(N, kBK4) * kBK4 > 2 * N) return false;
    if (numel > ((int64_t)12 << 30) || cdiv64(l.rows, kBM) > 65535 || P >= ((int64_t)1 << 31)) return false;
    if (Q == 1 ? (N % 8 != 0) : (Q % 64 != 0 || Q >= ((int64_t)1 << 31))) return false;
    l.bn = J <= 64 ? 64 : (cdiv64(J, 256) * 256 * 20 <= cdiv64(J, 128) * 128 * 23 ? 256 : 128);
    l.ks = (int)cdiv64(N, kBK4);
    auto a256 = [](size_t x) { return (x + 255) / 256 * 256; };
    // [max |X| at 0, the single slab maximum and the range flag at 256]
    // [fp16 images of X: shared by every product of one X] [this product's M^T,
    // ones, B images, column scales]
    size_t off = 512;
    l.off_img = off;
    off += 2 * a256((size_t)numel * 2);
    l.off_mt = off;
    off = a256(off + (size_t)N * J * 4);
    l.off_ones = off;
    off = a256(off + (size_t)J * 4);
    l.off_bimg = off;
    off = a256(off + (size_t)cdiv64(J, l.bn) * l.ks * 2 * l.bn * 128);
    l.off_colscale = off;
    off = a256(off + (size_t)J * 4);
    l.total = off;
    return true;
}
}  // namespace

size_t tc_ttm_workspace_bytes(int64_t P, int64_t N, int64_t Q, int64_t J) {
    TtmLayout l;
    return ttm_layout(P, N, Q, J, l) ? l.total : 0;
}

// The fp16 images of X (hi and lo at 512 and 512 + half) with one power-of-two
// scale from the sampled maximum, checked, redone exactly if the check fired
// (as in tc_prepare).  Shared by every product of one X.
int tc_ttm_images(const float* X, int64_t numel, void* ws, cudaStream_t stream, char* errbuf, size_t errlen) {
    if ((reinterpret_cast<uintptr_t>(X) & 15) != 0 || (reinterpret_cast<uintptr_t>(ws) & 255) != 0) {
        snprintf(errbuf, errlen, "the tensor-core mode-n product needs a 16-byte aligned X and a 256-byte aligned workspace");
        return MTTKRP_ERR_INVALID;
    }
    uint8_t* base = static_cast<uint8_t*>(ws);
    uint32_t* ymax = reinterpret_cast<uint32_t*>(base);
    uint32_t* slab = reinterpret_cast<uint32_t*>(base + 256);
    uint32_t* ovf = slab + 1;
    const size_t img_half = ((size_t)numel * 2 + 255) / 256 * 256;
    __half* img_hi = reinterpret_cast<__half*>(base + 512);
    __half* img_lo = reinterpret_cast<__half*>(base + 512 + img_half);
    cudaError_t e = cudaMemsetAsync(base, 0, 512, stream);
    if (e == cudaSuccess) {
        int64_t blocks = cdiv64(cdiv64(numel, kSlabUnit), 4);
        if (blocks > 152 * 8) blocks = 152 * 8;
        const int64_t nch = cdiv64(numel, kSampleChunk);
        int64_t sblocks = cdiv64(cdiv64(nch, nch > kSampleEvery ? kSampleEvery : 1), 8);
        if (sblocks > 152 * 8) sblocks = 152 * 8;
        slabsample_kernel<<<(unsigned)sblocks, 256, 0, stream>>>(X, 1, numel, slab, ymax);
        e = cudaGetLastError();
        if (e == cudaSuccess) {
            split_image_kernel<<<(unsigned)blocks, 256, 0, stream>>>(X, 1, numel, slab, ymax, img_hi, img_lo, ovf,
                                                                     nullptr);
            e = cudaGetLastError();
        }
        if (e == cudaSuccess) {
            slabmax_kernel<<<(unsigned)blocks, 256, 0, stream>>>(X, 1, numel, slab, ymax, ovf);
            e = cudaGetLastError();
        }
        if (e == cudaSuccess) {
            split_image_kernel<<<(unsigned)blocks, 256, 0, stream>>>(X, 1, numel, slab, ymax, img_hi, img_lo, nullptr,
                                                                     ovf);
            e = cudaGetLastError();
        }
    }
    if (e != cudaSuccess) {
        snprintf(errbuf, errlen, "mode-n product image pass: %s", cudaGetErrorString(e));
        return MTTKRP_ERR_CUDA;
    }
    return MTTKRP_OK;
}

int tc_ttm_run(const float* X, const float* M, float* T, int64_t P, int64_t N, int64_t Q, int64_t J, void* ws,
               cudaStream_t stream, char* errbuf, size_t errlen) {
    TtmLayout l;
    if (!ttm_layout(P, N, Q, J, l)) {
        snprintf(errbuf, errlen, "the tensor-core mode-n product does not take this shape");
        return MTTKRP_ERR_UNSUPPORTED;
    }
    const int rc = tc_ttm_images(X, P * N * Q, ws, stream, errbuf, errlen);
    if (rc != MTTKRP_OK) return rc;
    return tc_ttm_product(M, T, P, N, Q, J, ws, stream, errbuf, errlen);
}

// One product on images tc_ttm_images wrote into ws: M^T and its B images, then
// the image kernel with the mode-n-product epilogue.
int tc_ttm_product(const float* M, float* T, int64_t P, int64_t N, int64_t Q, int64_t J, void* ws,
                   cudaStream_t stream, char* errbuf, size_t errlen) {
    TtmLayout l;
    if (!ttm_layout(P, N, Q, J, l)) {
        snprintf(errbuf, errlen, "the tensor-core mode-n product does not take this shape");
        return MTTKRP_ERR_UNSUPPORTED;
    }
    PFN_cuTensorMapEncodeTiled_v12000 encode = encode_fn();
    uint32_t* status = tc_status_ptr();
    if (encode == nullptr || status == nullptr) {
        snprintf(errbuf, errlen, "tensor-map encoder or status word unavailable");
        return MTTKRP_ERR_CUDA;
    }
    uint8_t* base = static_cast<uint8_t*>(ws);
    uint32_t* ymax = reinterpret_cast<uint32_t*>(base);
    uint32_t* slab = reinterpret_cast<uint32_t*>(base + 256);
    float* mt = reinterpret_cast<float*>(base + l.off_mt);
    float* ones = reinterpret_cast<float*>(base + l.off_ones);
    float* bimg = reinterpret_cast<float*>(base + l.off_bimg);
    float* colscale = reinterpret_cast<float*>(base + l.off_colscale);
    const int64_t numel = P * N * Q;
    const size_t img_half = ((size_t)numel * 2 + 255) / 256 * 256;
    __half* img_hi = reinterpret_cast<__half*>(base + l.off_img);
    __half* img_lo = reinterpret_cast<__half*>(base + l.off_img + img_half);
    cudaError_t e;
    {
        int64_t blocks = cdiv64(J * N, 256);
        if (blocks > 152 * 8) blocks = 152 * 8;
        ttm_prep_kernel<<<(unsigned)blocks, 256, 0, stream>>>(M, J, N, mt, ones);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess) {
        ColScaleArgs c;
        memset(&c, 0, sizeof(c));
        c.ngroup = 1;
        c.gdim[0] = N;
        c.gfac[0] = mt;
        c.R = J;
        c.out = colscale;
        colscale_kernel<<<(unsigned)cdiv64(J, 32), 1024, 0, stream>>>(c);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess) {
        BImgArgs b;
        memset(&b, 0, sizeof(b));
        b.ngroup = 1;
        b.gdim[0] = N;
        b.gfac[0] = mt;
        b.R = J;
        b.J = N;
        b.Jq = N;
        b.BN = l.bn;
        b.KS = l.ks;
        b.jq_steps = l.ks;
        b.inner = 1;
        b.nblocks = cdiv64(J, l.bn) * l.ks;
        b.out = bimg;
        e = launch_bimage_f16<kBK4>(b, colscale, stream);
    }
    if (e != cudaSuccess) {
        snprintf(errbuf, errlen, "mode-n product preparation: %s", cudaGetErrorString(e));
        return MTTKRP_ERR_CUDA;
    }
    // tensor map of the natural images: (i, p) K-major for Q = 1, else (q, i, p)
    TcArgs args;
    memset(&args, 0, sizeof(args));
    cuuint64_t gdim[5];
    cuuint64_t gstride[4];
    cuuint32_t box[5], estr[5] = {1, 1, 1, 1, 1};
    int rank;
    for (int q = 0; q < kRoles; ++q) args.slot[q] = -1;
    if (Q == 1) {
        rank = 2;
        gdim[0] = (cuuint64_t)N;
        gdim[1] = (cuuint64_t)P;
        gstride[0] = (cuuint64_t)N * 2;
        box[0] = kBK4;
        box[1] = kBM;
        args.slot[kRoleJq] = 0;
        args.slot[kRoleI] = 1;
    } else {
        rank = 3;
        gdim[0] = (cuuint64_t)Q;
        gdim[1] = (cuuint64_t)N;
        gdim[2] = (cuuint64_t)P;
        gstride[0] = (cuuint64_t)Q * 2;
        gstride[1] = (cuuint64_t)N * Q * 2;
        box[0] = 64;
        box[1] = kBK4;
        box[2] = 1;
        args.slot[kRoleI] = 0;
        args.slot[kRoleJq] = 1;
        args.slot[kRolePP] = 2;
    }
    CUresult cr = encode(&args.ymap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, (cuuint32_t)rank, img_hi, gdim, gstride, box,
                         estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (cr == CUDA_SUCCESS)
        cr = encode(&args.ymap_lo, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, (cuuint32_t)rank, img_lo, gdim, gstride, box,
                    estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (cr != CUDA_SUCCESS) {
        snprintf(errbuf, errlen, "cuTensorMapEncodeTiled failed (%d)", (int)cr);
        return MTTKRP_ERR_CUDA;
    }
    args.rank = rank;
    args.bimg = bimg;
    args.gtab = ones;
    args.dst = T;
    args.dst_split_stride = 0;
    args.I = l.rows;
    args.R = J;
    args.npre = 1;
    args.pre_per_split = 1;
    args.nQ = 1;
    args.KS = l.ks;
    args.jq_steps = l.ks;
    args.ps = 1;
    args.batch_len = 1;
    args.y_box_bytes = (uint32_t)kBK4 * 2u * (uint32_t)kBM;
    args.ymax_bits = ymax;
    args.slab_bits = slab;
    args.slab_div = 1;
    args.slab_rows = 0;
    args.colscale = colscale;
    args.ttm_q = Q == 1 ? 0 : Q;
    args.g_ones = 1;
    args.status = status;
    // persistent: one CTA per SM, the row tiles of a column tile dealt out in
    // turn (the column tiles of one row tile run side by side and share its A
    // tiles through L2); the per-CTA start-up and the last tile's drain are paid
    // once per CTA instead of once per tile
    const int64_t gx = cdiv64(J, l.bn), ntiles = cdiv64(l.rows, kBM);
    int64_t gy = sm_count() / gx;
    if (gy < 1) gy = 1;
    if (gy > ntiles) gy = ntiles;
    args.tiles_y = ntiles;
    dim3 grid((unsigned)gx, (unsigned)gy, 1u);
    if (Q == 1)
        e = l.bn == 256 ? launch_img<256>(args, grid, stream)
          : l.bn == 128 ? launch_img<128>(args, grid, stream)
                        : launch_img<64>(args, grid, stream);
    else
        e = l.bn == 256 ? launch_img<256, false, true>(args, grid, stream)
          : l.bn == 128 ? launch_img<128, false, true>(args, grid, stream)
                        : launch_img<64, false, true>(args, grid, stream);
    if (e != cudaSuccess) {
        snprintf(errbuf, errlen, "tensor-core mode-n product launch: %s", cudaGetErrorString(e));
        return MTTKRP_ERR_CUDA;
    }
    return MTTKRP_OK;
}

uint32_t* tc_status_ptr() {
    static uint32_t* ptrs[64] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    if (ptrs[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
        ptrs[dev] = static_cast<uint32_t*>(p);
    }
    return ptrs[dev];
}

int tc_set_withhold_signal(int count) { return g_withhold_signal.exchange(count < 0 ? 0 : count); }

cudaError_t tc_read_and_clear_status(uint32_t* word) {
    cudaError_t err = cudaDeviceSynchronize();
    if (err != cudaSuccess) return err;
    err = cudaMemcpyFromSymbol(word, g_device_status, sizeof(uint32_t));
    if (err != cudaSuccess) return err;
    const uint32_t zero = 0;
    return cudaMemcpyToSymbol(g_device_status, &zero, sizeof(uint32_t));
}

}  // namespace mk
