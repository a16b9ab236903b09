// Blackwell (sm_100 family) tensor-core plumbing: tcgen05 MMA / TMEM,
// shared-memory matrix descriptors, mbarriers with bounded waits.
//
// Conventions used by the kernels:
//  * UMMA operands live in shared memory in the canonical layouts:
//      K-major, 128-byte swizzle: rows of 128 B, atoms of 8 rows (1 KB),
//        16-byte chunk c of row r stored at chunk c ^ (r & 7);
//        descriptor SBO = stride between 8-row groups, LBO unused;
//      MN-major, 128-byte swizzle: the same bytes read with M along the
//        128-byte row and K along rows (SBO = stride between 8-row groups
//        along K, LBO = stride between 128-byte column blocks along M);
//      MN-major, no swizzle: core matrices of 8 K-rows x 16 bytes
//        (LBO = stride between 8-row groups along K).
//  * every wait on an mbarrier gives up after a time limit, reports it in the
//    library's flag word and lets the caller unwind (no unbounded spin).
#pragma once

#include <stdint.h>

#include "common.cuh"

namespace mla {
namespace tc {

// ------------------------------------------------------------- descriptors

constexpr uint64_t kDefaultWaitLimitNs = 2000000000ull;

enum Swizzle : uint64_t { kSwizzleNone = 0, kSwizzle128B = 2, kSwizzle64B = 4, kSwizzle32B = 6 };

// Shared-memory matrix descriptor (sm_100 tcgen05 format).
MLA_DEVINLINE uint64_t smem_desc(uint32_t smem_addr, uint32_t lbo_bytes, uint32_t sbo_bytes,
                                 Swizzle swz) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((smem_addr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= 1ull << 46;                                  // descriptor version for sm_100
    d |= static_cast<uint64_t>(swz) << 61;
    return d;
}

// Instruction descriptor, kind::f8f6f4 with E4M3 x E4M3 -> F32.
// a_mn / b_mn select MN-major operands.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N, bool a_mn, bool b_mn) {
    return (1u << 4)                                  // D format: F32
           | (0u << 7) | (0u << 10)                   // A, B format: E4M3
           | (static_cast<uint32_t>(a_mn) << 15) | (static_cast<uint32_t>(b_mn) << 16)
           | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// Instruction descriptor, kind::f16 with BF16 x BF16 -> F32, both operands
// K-major.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
    return (1u << 4)                                  // D format: F32
           | (1u << 7) | (1u << 10)                   // A, B format: BF16
           | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// ------------------------------------------------------------------ tcgen05

MLA_DEVINLINE void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {   // whole warp
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n"
                 :: "r"(smem_u32(dst_smem)), "r"(ncols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
}
MLA_DEVINLINE void tmem_dealloc(uint32_t taddr, uint32_t ncols) {     // whole warp
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n"
                 :: "r"(taddr), "r"(ncols) : "memory");
}

MLA_DEVINLINE void mma_e4m3(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                            bool accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n"
        :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(static_cast<uint32_t>(accumulate))
        : "memory");
}

MLA_DEVINLINE void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                            bool accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
        :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(static_cast<uint32_t>(accumulate))
        : "memory");
}

// True in one lane of the calling (converged) warp: the lowest active lane,
// so the same lane every time the whole warp calls it.  tcgen05.mma and
// tcgen05.commit are issued by one thread; a warp that computes their
// operands together and elects the issuing lane keeps those operands
// warp-uniform.
MLA_DEVINLINE bool elect_one() {
    uint32_t pred = 0;
    asm volatile(
        "{\n .reg .pred p;\n elect.sync _|p, 0xffffffff;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(pred));
    return pred != 0;
}

// Arrives once on `bar` when every tcgen05.mma issued so far by this thread
// has completed.
MLA_DEVINLINE void mma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n"
                 :: "r"(smem_u32(bar)) : "memory");
}

MLA_DEVINLINE void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
MLA_DEVINLINE void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }

// Generic-proxy smem writes -> visible to the tensor core (async proxy).
MLA_DEVINLINE void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }

// 32 lanes x 16 columns of 32-bit TMEM cells: thread t gets lane (base + t).
MLA_DEVINLINE void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
// The same for 4 columns.
MLA_DEVINLINE void tmem_ld4(uint32_t taddr, uint32_t (&r)[4]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(taddr));
}
// M = 64 accumulators keep a warp's 16 rows in lanes 0-15 of its lane
// quadrant.  This load gives threads 0-15 those 16 lanes at columns
// col .. col + N - 1 and threads 16-31 the same lanes at columns
// col + kSplit .. (the 16x32bx2 shape), so both halves of the warp get data.
template <int kSplit>
MLA_DEVINLINE void tmem_ld_half8(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.16x32bx2.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8], %9;\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
        : "r"(taddr), "n"(kSplit));
}
template <int kSplit>
MLA_DEVINLINE void tmem_ld_half16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.16x32bx2.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16], %17;\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr), "n"(kSplit));
}

MLA_DEVINLINE void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory"); }

// 32 lanes x 16 columns: thread t writes lane (base + t).
MLA_DEVINLINE void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n"
        :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
           "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
           "r"(r[15])
        : "memory");
}
MLA_DEVINLINE void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory"); }

// ---------------------------------------------------------------- mbarrier

MLA_DEVINLINE void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" :: "r"(smem_u32(bar)), "r"(count) : "memory");
}
MLA_DEVINLINE void mbar_fence_init() { asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory"); }
MLA_DEVINLINE void mbar_arrive(uint64_t* bar) {
    asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.shared::cta.b64 st, [%0];\n}\n"
                 :: "r"(smem_u32(bar)) : "memory");
}
// Arrives on `bar` once all cp.async operations of this thread have landed.
MLA_DEVINLINE void mbar_arrive_cp_async(uint64_t* bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" :: "r"(smem_u32(bar)) : "memory");
}
MLA_DEVINLINE bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}
// Tests the phase without suspending the thread.
MLA_DEVINLINE bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}
// Arrives on `bar` and adds `bytes` to the transaction count its phase waits for.
MLA_DEVINLINE void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n"
                 :: "r"(smem_u32(bar)), "r"(bytes) : "memory");
}

// Bulk copy of `bytes` (a multiple of 16) from 16-byte aligned global memory
// to 16-byte aligned shared memory; completes as transaction bytes on `bar`.
MLA_DEVINLINE void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n"
        :: "r"(dst), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}

// Has L2 fetch every 128-byte line of the `kBytes` bytes at `row` (one
// prefetch per line, issued by the calling thread; nothing waits for them).
template <int kBytes>
MLA_DEVINLINE void prefetch_row_l2(const void* row) {
    const char* r = static_cast<const char*>(row);
#pragma unroll
    for (int o = 0; o < kBytes; o += 128)
        asm volatile("prefetch.global.L2 [%0];\n" :: "l"(r + o));
    // the line of the row's last byte (beyond the loop's lines when the row
    // starts past the middle of a line)
    asm volatile("prefetch.global.L2 [%0];\n" :: "l"(r + kBytes - 1));
}

// ----------------------------------------------------------------- clusters

MLA_DEVINLINE uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
    return r;
}
// All threads of all CTAs of the cluster meet; shared-memory writes made
// before it are visible to every CTA of the cluster after it.
MLA_DEVINLINE void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n"
                 "barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}
// The address of the same shared-memory variable in CTA `rank` of the cluster.
MLA_DEVINLINE uint32_t cluster_map(uint32_t smem_addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(r) : "r"(smem_addr), "r"(rank));
    return r;
}
MLA_DEVINLINE void st_cluster_f4(uint32_t cluster_addr, float4 v) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};\n"
                 :: "r"(cluster_addr), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w) : "memory");
}

MLA_DEVINLINE uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;\n" : "=l"(t));
    return t;
}

namespace {
// Default time limit of a bounded wait, in ns: one copy per translation unit
// that includes this header (the second in the constant bank, for
// mbar_wait_polled).  mla_debug_set_wait_limit changes the decode kernels'
// copies (tests use it to make a wait give up).
__device__ uint64_t g_wait_limit_ns = kDefaultWaitLimitNs;
__constant__ uint64_t c_wait_limit_ns = kDefaultWaitLimitNs;
}  // namespace

// Waits for the phase with the given parity to complete.  Gives up after
// `limit_ns` (0: the default limit above), or at once if *abort is already
// set; on giving up it sets *abort and the MLA_FLAG_WAIT_TIMEOUT flag and
// returns false.
MLA_DEVINLINE bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort, uint32_t* flags,
                             uint64_t limit_ns = 0) {
    if (mbar_try_wait(bar, parity)) return true;
    if (limit_ns == 0) limit_ns = g_wait_limit_ns;
    const uint64_t t0 = global_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (global_ns() - t0 > limit_ns) {
            *abort = 1;
            raise_flag(flags, MLA_FLAG_WAIT_TIMEOUT);
            return false;
        }
    }
}

// mbar_wait's contract, for warps that wait as a whole: the first test does
// not suspend, and the clock starts when it finds the phase incomplete; the
// thread then waits in try_wait.  A limit under kPollLimitNs (the test
// hook's) is checked between tests that do not suspend, so that it runs out
// on every wait that has to wait, however long the hardware lets a thread
// sleep in try_wait (a whole warp's try_wait can sleep through a wait of
// microseconds).  Measured on GB300 with 16-head CTAs: 33.2 us per batch-40
// call, against 34.0 with mbar_wait, 33.6 with try_wait's suspension bounded
// by a hint (0.5, 2 or 8 us) and 37.1 with a bounded try_wait as the first
// test.
constexpr uint64_t kPollLimitNs = 1000000;
// The part of the polled wait after a first test found the phase incomplete,
// out of line: one copy of the loop for every wait site (the 16-head decode
// kernel 77.4 -> 72.1 KB of code; the batch-40 call 30.66 vs 30.84 us on GB300).
static __device__ __noinline__ bool mbar_wait_polled_slow(uint64_t* bar, uint32_t parity, volatile int* abort,
                                                         uint32_t* flags) {
    const uint64_t lim = c_wait_limit_ns;
    const uint64_t t0 = global_ns();
    const bool poll = lim < kPollLimitNs;
    while (true) {
        if (poll ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (global_ns() - t0 > lim) {
            *abort = 1;
            raise_flag(flags, MLA_FLAG_WAIT_TIMEOUT);
            return false;
        }
    }
}
MLA_DEVINLINE bool mbar_wait_polled(uint64_t* bar, uint32_t parity, volatile int* abort, uint32_t* flags) {
    if (mbar_test_wait(bar, parity)) return true;
    return mbar_wait_polled_slow(bar, parity, abort, flags);
}

}  // namespace tc
}  // namespace mla
