// ptx_sm103.cuh -- inline-PTX wrappers for the Blackwell (sm_103a) asynchronous machinery used
// by the grouped GEMMs: mbarriers (with bounded waits), TMA tensor loads, tcgen05 tensor-memory
// allocation, tcgen05.mma (bf16 in, or block-scaled E4M3 / E2M1 in with the scales copied or
// stored into TMEM; fp32 accumulate in TMEM), tcgen05.commit, tcgen05.ld and tcgen05.st.
//
// Written from the public PTX ISA (tcgen05 / cp.async.bulk.tensor / mbarrier chapters). Every wait
// here is bounded: it gives up after kWaitTimeoutNs of wall time, sets MOE_DEV_TIMEOUT in the
// kernel's status word and raises the CTA's abort flag, so a broken pipeline ends the kernel with
// an error status instead of hanging the GPU.
#pragma once

#include <cuda.h>
#include <cstdint>

namespace moe {

constexpr unsigned long long kWaitTimeoutNs = 4000000000ull;  // 4 s

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------------------ programmatic dependent launch

// Blocks until the grids this one depends on (the previous kernel on the stream, when launched
// with programmatic stream serialization) have completed and their memory is visible. Returns at
// once when there is no such dependency. Every kernel calls it before its first global access.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Lets the next kernel on the stream be scheduled once every CTA of this grid has issued it (or
// exited); that kernel still waits in griddep_wait() for this grid to complete.
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Makes barrier initialisation visible to the async proxy (TMA, tcgen05) and to other threads.
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Waits for the phase with the given parity to complete. Returns false (after setting the status
// bit and the CTA abort flag) when the wait times out or another thread of the CTA has aborted.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          uint32_t* status, uint32_t timeout_bit,
                                          unsigned long long timeout_ns = kWaitTimeoutNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_timer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > timeout_ns) {
            atomicOr(status, timeout_bit);
            *abort_flag = 1;
            return false;
        }
    }
}

// ------------------------------------------------------- flags between CTAs of one grid

// Loads a counter with acquire semantics at GPU scope: writes released before the matching
// increment are visible to this thread after the load observes it.
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Adds to a counter with release semantics at GPU scope.
__device__ __forceinline__ void red_release_gpu_add(uint32_t* p, uint32_t v) {
    asm volatile("red.release.gpu.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Orders this thread's generic-proxy global accesses with the async proxy (TMA): after stores
// that another CTA's TMA will read, and after the acquire that precedes such a TMA read.
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// ---------------------------------------------------------------------------------------- TMA

__device__ __forceinline__ void tma_prefetch_descriptor(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2-D tiled bulk tensor load global -> shared; completion is signalled on `bar` as transaction
// bytes. x is the innermost (contiguous) coordinate in elements, y the row.
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int32_t x,
                                            int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(smem_addr(smem_dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

// The same for a 3-D tensor map: box element (x, y, z) of the box at coordinates (x, y, z).
__device__ __forceinline__ void tma_load_3d(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int32_t x,
                                            int32_t y, int32_t z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
        ::"r"(smem_addr(smem_dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
        : "memory");
}

// Asks L2 to fetch the 128-byte line holding `p` (no register result, no wait).
__device__ __forceinline__ void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// 1-D bulk copy global -> shared of `bytes` (a multiple of 16; both addresses 16-byte aligned),
// completion signalled on `bar` as transaction bytes.
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_addr(smem_dst)), "l"(reinterpret_cast<uint64_t>(gsrc)), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// ------------------------------------------------------------------------------ tensor memory

// Allocates `ncols` TMEM columns (power of two, >= 32) for this CTA; the whole warp must execute
// it. The TMEM address is written to *slot (shared memory).
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(slot)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish_alloc_permit() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tcgen05_fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tcgen05_fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ------------------------------------------------------------------------------------ tcgen05

// Shared-memory matrix descriptor for a K-major operand tile written by TMA with 128-byte
// swizzling: rows of 128 bytes (64 bf16 along K), 8-row swizzle atoms of 1024 bytes stacked along
// M/N. Fields: start address >> 4 [0,14), leading-dimension byte offset >> 4 [16,30) (not used by
// swizzled K-major layouts), stride-dimension byte offset >> 4 [32,46) = 1024 B between 8-row
// groups, descriptor version 1 at [46,48), base offset 0 (atoms are 1024-byte aligned), swizzle
// mode 2 = 128-byte swizzle at [61,64).
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(16u >> 4) << 16;
    d |= static_cast<uint64_t>(1024u >> 4) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    d |= static_cast<uint64_t>(2u) << 61;
    return d;
}

// The same for an MN-major operand tile (M or N contiguous), as TMA writes it from boxes of
// 64 (M or N) x rows-of-K with 128-byte swizzling: each box is a column of 8-row swizzle atoms
// (one K row = 64 M/N values = 128 bytes). Canonical layout ((64, m), (8, k)): the leading-
// dimension byte offset is the distance between 64-wide M/N blocks (one box, mn_block_bytes), the
// stride-dimension byte offset the distance between 8-row K groups (1024 bytes).
__device__ __forceinline__ uint64_t sw128_mnmajor_desc(uint32_t saddr, uint32_t mn_block_bytes) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((mn_block_bytes >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>(1024u >> 4) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    d |= static_cast<uint64_t>(2u) << 61;
    return d;
}

// Instruction descriptor of tcgen05.mma .kind::f16: D fp32 (bits [4,6) = 1), A and B bf16
// (bits [7,10) and [10,13) = 1), A / B major-ness at bits 15 / 16 (0 = K-major, 1 = MN-major),
// N >> 3 at [17,23), M >> 4 at [24,29).
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn_major = false,
                                                      bool b_mn_major = false) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
           (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]^T for one M x N x 16 step, issued by a single thread.
__device__ __forceinline__ void mma_bf16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// ------------------------------------------------------------------- block-scaled (MXFP8) MMA
//
// Scale factors live in TMEM. A 512-byte shared-memory chunk holds the UE8M0 scales of 128 rows
// (of A, or of B's N dimension) for four consecutive 32-element K blocks: row r, block k at byte
// 16 * (r % 32) + 4 * (r / 32) + k. tcgen05.cp .32x128b.warpx4 copies it as 32 rows of 16 bytes
// into columns c .. c+3 of every 32-lane quarter of TMEM, so the scale of row r sits in column
// c + r / 32, byte k, of lane r % 32 of each quarter; the MMA's scale-factor id picks byte k. A
// 256-row operand (B with N > 128) takes two chunks in columns c .. c+7. The same TMEM layout can
// be written by four warps instead (one per lane quarter, tmem_st_32cols): lane l of each quarter
// stores the chunk's 16 bytes at 16 l into columns c .. c+3.

// Shared-memory descriptor of one such chunk: no swizzle, 8-row core matrices of 16-byte rows
// stacked 128 bytes apart (stride-dimension byte offset 128), descriptor version 1.
__device__ __forceinline__ uint64_t sf_chunk_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(128u >> 4) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    return d;
}

// Copies one 512-byte scale chunk from shared memory to TMEM columns taddr .. taddr+3 of all four
// lane quarters. Issued by one thread; ordered before the tcgen05.mma it issues afterwards.
__device__ __forceinline__ void tmem_cp_scale_chunk(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// Instruction descriptor of tcgen05.mma .kind::mxf8f6f4 with A and B E4M3 (format 0 at [7,10) and
// [10,13)), both K-major, N >> 3 at [17,23), UE8M0 scales (bit 23), M >> 4 at [24,29). The
// scale-factor ids (B at [4,6), A at [29,31)) are added per K step by mxf8_ids().
__host__ __device__ constexpr uint32_t idesc_mxf8_e4m3(int M, int N) {
    return (static_cast<uint32_t>(N >> 3) << 17) | (1u << 23) | (static_cast<uint32_t>(M >> 4) << 24);
}

__host__ __device__ constexpr uint32_t mxf8_ids(int k) {
    return (static_cast<uint32_t>(k) << 4) | (static_cast<uint32_t>(k) << 29);
}

// D[tmem] (+)= (A * 2^sfa) (B * 2^sfb)^T for one M x N x 32 step of E4M3 operands with one UE8M0
// scale per row and 32 K elements (scale_vec::1X), issued by a single thread.
__device__ __forceinline__ void mma_mxf8_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
        ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// Instruction descriptor of tcgen05.mma .kind::mxf4nvf4 with A and B E2M1 (format 1 at [7,10) and
// [10,13)), both K-major, N >> 3 at [17,23), UE4M3 scales (bit 23 clear), M >> 4 at [24,29); the
// scale-factor ids stay 0 (each MMA reads all four bytes of its scale column).
__host__ __device__ constexpr uint32_t idesc_nvf4(int M, int N) {
    return (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// D[tmem] (+)= (A * sfa) (B * sfb)^T for one M x N x 64 step of packed E2M1 operands (two per
// byte, low nibble first) with one UE4M3 scale per row and 16 K elements (scale_vec::4X): a
// 512-byte scale chunk in TMEM holds the four scales of each of 128 rows for this step.
__device__ __forceinline__ void mma_nvf4_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
        ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// Arrives once on `bar` when every tcgen05.mma issued so far by this thread has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_addr(bar))
                 : "memory");
}

// Loads 32 consecutive fp32 columns of this thread's TMEM lane (shape 32x32b, 32 repetitions):
// thread i of the warp reads lane (taddr.lane + i), columns taddr.col .. taddr.col + 31.
__device__ __forceinline__ void tmem_ld_32cols(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

// Stores 32 consecutive 32-bit columns of this thread's TMEM lane (shape 32x32b, 32 repetitions):
// thread i of the warp writes lane (taddr.lane + i), columns taddr.col .. taddr.col + 31. The warp
// may only address its own 32-lane quarter of TMEM (warp index % 4).
__device__ __forceinline__ void tmem_st_32cols(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};"
        ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
          "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
          "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
          "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

// Waits until this thread's outstanding tcgen05.st have written TMEM.
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Waits for this thread's outstanding tcgen05.ld; the register operands tie the loaded values to
// the wait so the compiler cannot move their uses above it.
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                   "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                   "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}

// Orders a second register array after a preceding tmem_ld_wait (no instruction emitted).
__device__ __forceinline__ void tmem_ld_tie(uint32_t (&r)[32]) {
    asm volatile(""
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                   "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                   "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}

}  // namespace moe
