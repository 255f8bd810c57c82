// Inline-PTX helpers for sm_103a: mbarriers with bounded waits, TMA (bulk tensor)
// loads, cluster barriers and distributed shared memory, and the warp-level
// bf16 tensor-core MMA.  Every wait here has a time limit: a wait that gives up
// records Q4K_DEV_TIMEOUT in the caller's status word and returns false.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace q4k {

constexpr unsigned int kDevTimeout = 1u;         // status bit: a bounded wait gave up
constexpr unsigned int kDevRouting = 2u;         // status bit: a reused routing was made for another call shape
// Written by the routing kernel after the tile count, with (E, item count): a
// call that reuses the routing checks that it was made for its own shape.
constexpr int kRoutingStamp = 0x5134524B;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// SwiGLU of one element of a routed expert's feed-forward layer, rounded once
// to bf16 (nearest, ties to even): silu(g) * u with silu(g) = g / (1 + e^-g).
// e^-g = 2^(-g log2 e) and the reciprocal come from the approximate ex2 and rcp
// instructions (a few fp32 ulps together, far below the bf16 rounding that
// follows; the down projection reads bf16).  For g below about -88, e^-g is +inf
// and its reciprocal +0, so h is a signed zero, the limit of silu.  Seven
// instructions: the tensor-core kernels' epilogue competes for issue slots with
// their dequantizing warps.
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ uint16_t swiglu_bf16(float g, float u) {
    constexpr float kLog2e = 1.4426950408889634f;
    const float h = g * rcp_approx(1.0f + ex2_approx(-kLog2e * g)) * u;
    return __bfloat16_as_ushort(__float2bfloat16_rn(h));
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking test of the phase with the given parity.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase with the given parity to complete.  Gives up after
// limit_ns, sets the timeout bit in *status and returns false.  A limit under
// 1 us (a test of the give-up path) tests the phase once, without blocking, and
// gives up at once if it has not completed; limits under 100 us are checked on
// every retry.
__device__ __forceinline__ bool mbar_wait_limit(uint32_t bar, uint32_t parity, unsigned int *status,
                                                unsigned long long limit_ns) {
    if (limit_ns < 1000ull) {
        if (mbar_test_wait(bar, parity)) return true;
        atomicOr(status, kDevTimeout);
        return false;
    }
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    const uint32_t every = limit_ns < 100000ull ? 0u : 63u;
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & every) == 0 && global_timer_ns() - t0 > limit_ns) {
            atomicOr(status, kDevTimeout);
            return false;
        }
    }
}

// mbar_wait_limit with the standard limit, kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, unsigned int *status) {
    return mbar_wait_limit(bar, parity, status, kWaitLimitNs);
}

// Whether the routing header hdr = {tile count, E, items, stamp} in the workspace
// was written for E experts and n_items items; if not, thread 0 of CTA 0 records
// kDevRouting in *status (the caller then leaves before touching the routing).
__device__ __forceinline__ bool routing_matches(const int *hdr, int E, int n_items, unsigned int *status) {
    const bool ok = __ldg(hdr + 1) == E && __ldg(hdr + 2) == n_items && __ldg(hdr + 3) == kRoutingStamp;
    if (!ok && threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) atomicOr(status, kDevRouting);
    return ok;
}

// ---------------------------------------------------------------------- TMA
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *m) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

// 2-D tiled bulk-tensor load into this CTA's shared memory, completion counted
// in bytes on `bar`.  c0 is the innermost coordinate (elements).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *m, int32_t c0, int32_t c1, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

// Orders this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (TMA / tensor core) accesses to the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------ cluster
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// address of the same shared-memory variable in CTA `rank` of this cluster
__device__ __forceinline__ uint32_t map_shared_rank(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

// Split cluster barrier: arrive (release) early, wait (acquire) later.
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
// Arrive without ordering memory: for a phase that only marks progress (the
// caller's stores were already released by other means).
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

__device__ __forceinline__ void st_shared_cluster_f32(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// Arrive (release, cluster scope) on an mbarrier of another CTA of the cluster
// (addr from map_shared_rank).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(addr) : "memory");
}

// mbar_wait with cluster-scope acquire (the arrivals come from other CTAs of the
// cluster) and a caller-chosen limit.
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, unsigned int *status,
                                                  unsigned long long limit_ns) {
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 0;; ++i) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
        if (ok) return true;
        if ((i & 63u) == 63u && global_timer_ns() - t0 > limit_ns) {
            atomicOr(status, kDevTimeout);
            return false;
        }
    }
}

__device__ __forceinline__ float ld_shared_cluster_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

// -------------------------------------------------------------- bit helpers
__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
    // (a & b) | c
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// ------------------------------------------------------------------ NVFP4
// Eight e2m1 codes of one 32-bit value word (weight 2i in the low nibble of byte
// i) -> four bf16 pairs in natural order, each the exact e2m1 value.  The
// magnitudes come from two 8-entry byte tables selected by the codes' low three
// bits (bf16 high bytes 00 3F 3F 3F 40 40 40 40, low bytes 00 00 80 C0 00 40 80
// C0: 0, 0.5, 1, 1.5, 2, 3, 4, 6); each code's sign bit moves to bit 7 of its
// high byte.
__device__ __forceinline__ void e2m1x8_to_bf16(uint32_t w, uint32_t &p01, uint32_t &p23, uint32_t &p45,
                                               uint32_t &p67) {
    const uint32_t m = w & 0x77777777u;
    const uint32_t w4 = w << 4;
    const uint32_t sa = prmt(w4, w, 0x5140u), sb = prmt(w4, w, 0x7362u);  // element k's sign -> bit 7 of byte k
    const uint32_t hia = prmt(0x3F3F3F00u, 0x40404040u, m) | (sa & 0x80808080u);
    const uint32_t loa = prmt(0xC0800000u, 0xC0804000u, m);
    const uint32_t hib = prmt(0x3F3F3F00u, 0x40404040u, m >> 16) | (sb & 0x80808080u);
    const uint32_t lob = prmt(0xC0800000u, 0xC0804000u, m >> 16);
    p01 = prmt(loa, hia, 0x5140u);
    p23 = prmt(loa, hia, 0x7362u);
    p45 = prmt(lob, hib, 0x5140u);
    p67 = prmt(lob, hib, 0x7362u);
}

// e4m3 (finite variant) -> fp32, exact (through the exact e4m3 -> fp16 conversion)
__device__ __forceinline__ float e4m3_to_f32(uint32_t b) {
    const __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)(b & 0xFFu), __NV_E4M3);
    return __half2float(__half(h));
}

// ------------------------------------------------------------- tensor core
// D = A(16x16 bf16, row) * B(16x8 bf16, col) + C, fp32 accumulate.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1,
                                               const float (&c)[4]) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%10, %11, %12, %13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]),
          "f"(c[3]));
}

// D = A(16x16 fp16, row) * B(16x8 fp16, col) + C, fp32 accumulate.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1,
                                              const float (&c)[4]) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%10, %11, %12, %13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]),
          "f"(c[3]));
}

// ------------------------------------------------- tcgen05 / tensor memory
// Descriptor of a K-major bf16 operand tile in shared memory laid out in the
// canonical 128-byte-swizzle form: rows of 64 bf16 (128 bytes), 8-row atoms of
// 1024 bytes stacked along M/N (stride byte offset 1024), 16-byte chunks of row r
// XOR-permuted by r % 8.  Fields (PTX ISA, tcgen05 shared memory descriptor):
// [0,14) start address >> 4, [16,30) leading byte offset >> 4 (unused for
// swizzled K-major: 1), [32,46) stride byte offset >> 4, [46,49) fixed 0b001,
// [49,52) base offset (0: atoms are 1024-byte aligned), [52] LBO mode 0,
// [61,64) swizzle mode 2 = 128-byte swizzle.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t smem_addr) {
    uint64_t d = 0;
    d |= (uint64_t)((smem_addr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor of tcgen05.mma .kind::f16 (PTX ISA table): [4,6) D
// format 1 = f32, [7,10) A format 1 = bf16, [10,13) B format 1 = bf16, [15] A
// K-major 0, [16] B K-major 0, [17,23) N >> 3, [24,29) M >> 4.
__host__ __device__ constexpr uint32_t umma_idesc_bf16_f32(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Allocates `ncols` tensor-memory columns (a power of two >= 32) for this CTA;
// the base address is written to shared memory at `dst`.  Whole warp.
__device__ __forceinline__ void tmem_alloc(uint32_t dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, both K-major; accumulate when `acc` != 0.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(acc)
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T: row i of A in tensor-memory lane i, its K
// elements packed two per 32-bit column (16 elements: 8 columns from a_tmem);
// B in shared memory, K-major.  Accumulate when `acc` != 0.
__device__ __forceinline__ void umma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                             uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
        ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(acc)
        : "memory");
}

// 4 / 8 / 16 consecutive 32-bit columns of this thread's tensor-memory lane from
// registers (whole warp; the warp's lane quarter); tmem_st_wait() completes them.
__device__ __forceinline__ void tmem_st4(uint32_t taddr, const uint32_t (&v)[4]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};"
                 ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3])
                 : "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&v)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
                 ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
                 : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
                 "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
                 ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
                 "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
                 : "memory");
}
template <int NC>
__device__ __forceinline__ void tmem_st(uint32_t taddr, const uint32_t (&v)[NC]) {
    if constexpr (NC == 4) {
        tmem_st4(taddr, v);
    } else if constexpr (NC == 8) {
        tmem_st8(taddr, v);
    } else {
        static_assert(NC == 16, "4, 8 or 16 columns");
        tmem_st16(taddr, v);
    }
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Arrive on `bar` once every tcgen05 operation this thread issued has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 consecutive fp32 columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
          "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
          "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// ------------------------------------------------ programmatic dependent launch
// Every kernel of the library is launched with programmatic stream
// serialization, so it may start while the previous kernel in the stream is
// still draining.  pdl_wait blocks until that kernel has completed and its
// memory is visible; each kernel calls it before its first global-memory
// access.  pdl_trigger lets the next kernel in the stream start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ uint32_t elect_one() {
    uint32_t pred = 0;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "elect.sync _|p, 0xffffffff;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(pred));
    return pred;
}


// ------------------------------------------- Q4_K -> tensor-core operand
// packed fp32 pairs: a * b + c and a + b, each element rounded once
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;"
        : "=l"(d)
        : "l"(*reinterpret_cast<unsigned long long *>(&a)), "l"(*reinterpret_cast<unsigned long long *>(&b)),
          "l"(*reinterpret_cast<unsigned long long *>(&c)));
    return *reinterpret_cast<float2 *>(&d);
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
    unsigned long long d;
    asm("add.rn.f32x2 %0, %1, %2;"
        : "=l"(d)
        : "l"(*reinterpret_cast<unsigned long long *>(&a)), "l"(*reinterpret_cast<unsigned long long *>(&b)));
    return *reinterpret_cast<float2 *>(&d);
}

// The scales of one 64-weight group of a Q4_K block: sub-block 2g (low nibbles,
// d sc and -dmin m as fp32 pairs) and 2g+1 (high nibbles).
struct GroupScales {
    float2 ds0, dmn0, ds1, dmn1;
};
__device__ __forceinline__ GroupScales group_scales(float dsc0, float dm0, float dsc1, float dm1) {
    return {make_float2(dsc0, dsc0), make_float2(-dm0, -dm0), make_float2(dsc1, dsc1), make_float2(-dm1, -dm1)};
}

// One 32-bit word of codes (4 bytes = elements e..e+3 of sub-blocks 2g and 2g+1)
// -> the bf16 operand pairs (e, e+1), (e+2, e+3) of each sub-block, each weight
// the round-to-nearest-even bf16 of the fp32 dequantized value
// fl32(q * d sc - dmin m): q * d sc is exact inside the FMA (21 significant
// bits), so the fp32 value is the one rounding of the exact weight, the same
// value the standalone dequantization writes.  The nibbles become the floats
// 2^23 + q by one byte permute each; q = that - 2^23 exactly.
__device__ __forceinline__ void q4k_word_to_bf16(uint32_t w, const GroupScales &c, uint32_t &lo01, uint32_t &lo23,
                                                 uint32_t &hi01, uint32_t &hi23) {
    const uint32_t lw = w & 0x0F0F0F0Fu, hw = (w >> 4) & 0x0F0F0F0Fu;
    const float2 k23n = make_float2(-8388608.0f, -8388608.0f);
    uint32_t out[4];
#pragma unroll
    for (int pr = 0; pr < 2; ++pr) {
        const float l0 = __uint_as_float(prmt(lw, 0x4B000000u, 0x7650u + 2 * pr));
        const float l1 = __uint_as_float(prmt(lw, 0x4B000000u, 0x7651u + 2 * pr));
        const float h0 = __uint_as_float(prmt(hw, 0x4B000000u, 0x7650u + 2 * pr));
        const float h1 = __uint_as_float(prmt(hw, 0x4B000000u, 0x7651u + 2 * pr));
        const float2 wl = fma2(add2(make_float2(l0, l1), k23n), c.ds0, c.dmn0);
        const float2 wh = fma2(add2(make_float2(h0, h1), k23n), c.ds1, c.dmn1);
        const __nv_bfloat162 bl = __floats2bfloat162_rn(wl.x, wl.y), bh = __floats2bfloat162_rn(wh.x, wh.y);
        out[pr] = *reinterpret_cast<const uint32_t *>(&bl);
        out[2 + pr] = *reinterpret_cast<const uint32_t *>(&bh);
    }
    lo01 = out[0], lo23 = out[1], hi01 = out[2], hi23 = out[3];
}

}  // namespace q4k
