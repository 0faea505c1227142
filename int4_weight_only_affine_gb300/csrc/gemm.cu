// f16_gemm: dense half GEMM of the prefill path, Y[M][N] = X[M][K] * W16[K][N].
//
// "The inference engine - Mojo 1.0 on Metal", "Crossing Mojo 1.0": after the
// dequantise-once step prefill runs a half-precision GEMM on the transposed
// scratch; the same page credits hoisting tile-edge guards out of the GEMM
// hot loop.  Here the hot loop has no edge guards at all: tensor-memory
// copies zero-fill out-of-range rows/columns and only the epilogue masks.
//
// sm_103a design:
//  * Persistent grid (one CTA per SM), static tile schedule over 128 x 256
//    output tiles, m-fastest so CTAs in flight share W16 columns in L2.
//  * Warp 0: one thread issues TMA copies (128B-swizzled boxes) of the A
//    tile (X, K-major, 128 x 64) and B tile (W16, N-major, 64 x 256 as four
//    64 x 64 boxes) into a 4-stage shared-memory ring (mbarrier tx counts).
//  * Warp 1: allocates 512 TMEM columns (two 128 x 256 fp32 accumulators)
//    and one thread issues tcgen05.mma.kind::f16 (M=128, N=256, K=16; four
//    per 64-k stage), releasing each stage with tcgen05.commit.
//  * Warps 2-5: epilogue.  Each reads its 32 TMEM lanes (tcgen05.ld), rounds
//    to binary16 and stores; the accumulator is released as soon as it has
//    been read, so the next tile's MMAs overlap the stores.
//  * Every mbarrier wait is bounded (2 s); on expiry the kernel records
//    W4_ERR_TIMEOUT in a device flag, drains its own copies and MMAs, frees
//    TMEM and returns.
#include <cuda.h>

#include "common.cuh"

namespace w4a16 {


namespace {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_TILE = BM * BK * 2;     // 16 KB
constexpr int B_BOX = BK * 64 * 2;      // 8 KB: 64 k rows x 64 n
constexpr int B_TILE = BK * BN * 2;     // 32 KB
constexpr int STAGE_BYTES = A_TILE + B_TILE;
constexpr int NUM_THREADS = 192;
constexpr int TMEM_COLS = 2 * BN;
constexpr size_t SMEM_BYTES = 1024 + (size_t)STAGES * STAGE_BYTES + 256;
// Shared-memory matrix descriptor (sm_100 family): start address, leading and
// stride byte offsets (>> 4), descriptor version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((addr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor, kind::f16: fp32 accumulate, A and B binary16, A
// K-major, B MN-major, N = 256, M = 128.
constexpr uint32_t kInstrDesc = (1u << 4)                 // D format: f32
                                | (0u << 7) | (0u << 10)  // A, B: f16
                                | (0u << 15)              // A K-major
                                | (1u << 16)              // B MN-major
                                | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);

__device__ __forceinline__ void mma_f16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t accum) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(kInstrDesc), "r"(accum));
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
          "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
          "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t pack_half2(uint32_t a, uint32_t b) {
    const __half2 h = __floats2half2_rn(__uint_as_float(a), __uint_as_float(b));
    return *reinterpret_cast<const uint32_t *>(&h);
}

// The B tile of a stage: 64 k rows x BN columns of W16 as BN / 64 boxes of
// 64 x 64 (128-byte swizzle), box j at sb + j * B_BOX.  With b3d the tensor
// map views W16 as [N / 64][K][64] and one copy brings all BN / 64 boxes
// (each k row's 512 bytes contiguous in memory: fewer, longer DRAM bursts).
__device__ __forceinline__ void load_b_tile(uint32_t sb, const CUtensorMap *map, int n0, int k0, uint32_t bar,
                                            int b3d) {
    if (b3d) {
        tma_load_3d(sb, map, 0, k0, n0 / 64, bar);
    } else {
#pragma unroll
        for (int j = 0; j < BN / 64; ++j) tma_load_2d(sb + j * B_BOX, map, n0 + 64 * j, k0, bar);
    }
}

// pdl: launched as a programmatic dependent.  The kernel releases the next
// one at once, sets up and copies the weight (B) tiles of its first stages
// before waiting for the previous kernel; the activation (A) copies, and so
// every read of data the previous kernel may write and every output store,
// come after the wait.
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tma_a, const __grid_constant__ CUtensorMap tma_b,
                uint16_t *__restrict__ y, int M, int N, int K, int pdl, int b3d) {
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment for the 128-byte swizzle atoms.
    const uint32_t raw = (uint32_t)__cvta_generic_to_shared(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    const uint32_t bar0 = base + STAGES * STAGE_BYTES;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto accf_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + a); };
    auto acce_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + 2 + a); };
    const uint32_t done_bar = bar0 + 8u * (2 * STAGES + 4);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + STAGES * STAGE_BYTES + 8 * (2 * STAGES + 5));

    pdl_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tiles_m = (M + BM - 1) / BM, tiles_n = (N + BN - 1) / BN;
    const int ntiles = tiles_m * tiles_n;
    const int nk = (K + BK - 1) / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(accf_bar(a), 1);
            mbar_init(acce_bar(a), 4);
        }
        mbar_init(done_bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(&tma_a) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(&tma_b) : "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         (uint32_t)__cvta_generic_to_shared(tmem_slot)),
                     "r"(TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer ----------------
            uint32_t issued_ph = 0, issued_any = 0;
            int it = 0;
            bool ok = true;
            int pre = 0;  // first-tile stages whose B copies precede the dependency wait
            if (pdl && blockIdx.x < ntiles) {
                const int m0 = (blockIdx.x % tiles_m) * BM, n0 = (blockIdx.x / tiles_m) * BN;
                pre = nk < STAGES ? nk : STAGES;
                for (int kb = 0; kb < pre; ++kb) {  // fresh slots: no empty wait
                    mbar_expect_tx(full_bar(kb), STAGE_BYTES);
                    const uint32_t sb = base + kb * STAGE_BYTES + A_TILE;
                    load_b_tile(sb, &tma_b, n0, kb * BK, full_bar(kb), b3d);
                    issued_any |= 1u << kb;
                }
                pdl_wait();
                for (int kb = 0; kb < pre; ++kb) tma_load_2d(base + kb * STAGE_BYTES, &tma_a, kb * BK, m0, full_bar(kb));
                it = pre;
            } else if (pdl) {
                pdl_wait();
            }
            for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
                const int m0 = (t % tiles_m) * BM, n0 = (t / tiles_m) * BN;
                for (int kb = (t == (int)blockIdx.x) ? pre : 0; kb < nk; ++kb, ++it) {
                    const int s = it % STAGES;
                    const uint32_t ph = (it / STAGES) & 1;
                    if (!mbar_wait(empty_bar(s), ph ^ 1)) {
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(full_bar(s), STAGE_BYTES);
                    const uint32_t sa = base + s * STAGE_BYTES;
                    const uint32_t sb = sa + A_TILE;
                    tma_load_2d(sa, &tma_a, kb * BK, m0, full_bar(s));
                    load_b_tile(sb, &tma_b, n0, kb * BK, full_bar(s), b3d);
                    issued_ph = (issued_ph & ~(1u << s)) | (ph << s);
                    issued_any |= 1u << s;
                }
            }
            // Drain: every copy this thread issued has landed before exit.
            for (int s = 0; s < STAGES; ++s)
                if (issued_any & (1u << s)) mbar_wait(full_bar(s), (issued_ph >> s) & 1);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            int it = 0, tc = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x, ++tc) {
                const int acc = tc & 1;
                const uint32_t aph = (tc >> 1) & 1;
                if (!mbar_wait(acce_bar(acc), aph ^ 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t dst = tmem + acc * BN;
                for (int kb = 0; kb < nk; ++kb, ++it) {
                    const int s = it % STAGES;
                    const uint32_t ph = (it / STAGES) & 1;
                    if (!mbar_wait(full_bar(s), ph)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = base + s * STAGE_BYTES;
                    const uint32_t sb = sa + A_TILE;
#pragma unroll
                    for (int ks = 0; ks < BK / 16; ++ks) {
                        const uint64_t ad = smem_desc(sa + ks * 32, 16, 1024);
                        const uint64_t bd = smem_desc(sb + ks * 2048, B_BOX, 1024);
                        mma_f16(dst, ad, bd, (kb | ks) != 0);
                    }
                    mma_commit(empty_bar(s));
                }
                if (!ok) break;
                mma_commit(accf_bar(acc));
            }
            mma_commit(done_bar);
            mbar_wait(done_bar, 0);
        }
    } else {
        // ---------------- epilogue: warps 2..5 ----------------
        const int quad = warp & 3;  // TMEM lanes 32*quad .. 32*quad+31
        int tc = 0;
        for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++tc) {
            const int m0 = (t % tiles_m) * BM, n0 = (t / tiles_m) * BN;
            const int acc = tc & 1;
            const uint32_t aph = (tc >> 1) & 1;
            if (!mbar_wait(accf_bar(acc), aph)) break;
            tc_fence_after();
            const int row = m0 + quad * 32 + lane;
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t r[32];
                tmem_ld32(tmem + ((uint32_t)(quad * 32) << 16) + acc * BN + c * 32, r);
                if (c == BN / 32 - 1) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(acce_bar(acc));
                }
                if (row < M) {
                    uint16_t *dst = y + (size_t)row * N + n0 + c * 32;
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        if (n0 + c * 32 + 8 * v < N) {
                            uint4 o;
                            o.x = pack_half2(r[8 * v + 0], r[8 * v + 1]);
                            o.y = pack_half2(r[8 * v + 2], r[8 * v + 3]);
                            o.z = pack_half2(r[8 * v + 4], r[8 * v + 5]);
                            o.w = pack_half2(r[8 * v + 6], r[8 * v + 7]);
                            *reinterpret_cast<uint4 *>(dst + 8 * v) = o;
                        }
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS));
    }
}

// ---------------------------------------------------------------------------
// CTA-pair variant (cta_group::2): a cluster of two CTAs computes a 256 x 256
// tile.  Each CTA loads its own 128 rows of X and its own 128 columns of W16
// (half the operand bytes per SM of the single-CTA tile); the leader CTA
// issues tcgen05.mma.cta_group::2 (M=256, N=256, K=16), which reads A and B
// from both CTAs' shared memory and accumulates rows 0-127 in the leader's
// TMEM and rows 128-255 in the peer's.  Both CTAs' copies complete on the
// leader's stage barrier; commits are multicast to both CTAs; both CTAs'
// epilogue warps release an accumulator by arriving on the leader's barrier.
// ---------------------------------------------------------------------------
constexpr int ST2 = 6;
constexpr int A2_TILE = 128 * BK * 2;      // 16 KB: this CTA's 128 rows
constexpr int B2_HALF = BK * 128 * 2;      // 16 KB: this CTA's 128 columns
constexpr int STAGE2_BYTES = A2_TILE + B2_HALF;
constexpr size_t SMEM2_BYTES = 1024 + (size_t)ST2 * STAGE2_BYTES + 256;
constexpr uint32_t kInstrDesc2 = (1u << 4) | (0u << 7) | (0u << 10) | (0u << 15) | (1u << 16) |
                                 ((uint32_t)(256 >> 3) << 17) | ((uint32_t)(256 >> 4) << 24);

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                                 uint32_t leader_bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
        "%3}], [%4];" ::"r"(dst),
        "l"(map), "r"(c0), "r"(c1), "r"(leader_bar)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap *map, int c0, int c1, int c2,
                                                 uint32_t leader_bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
        "%3, %4}], [%5];" ::"r"(dst),
        "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(leader_bar)
        : "memory");
}

// This CTA's 128 columns of a pair's B tile (two 64 x 64 boxes; with b3d one
// copy of the [N / 64][K][64] view, as load_b_tile).
__device__ __forceinline__ void load_b_half_pair(uint32_t sb, const CUtensorMap *map, int n0, int k0,
                                                 uint32_t leader_bar, int b3d) {
    if (b3d) {
        tma_load_3d_pair(sb, map, 0, k0, n0 / 64, leader_bar);
    } else {
        tma_load_2d_pair(sb, map, n0, k0, leader_bar);
        tma_load_2d_pair(sb + B_BOX, map, n0 + 64, k0, leader_bar);
    }
}

__device__ __forceinline__ void mma_f16_pair(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t accum) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(kInstrDesc2), "r"(accum));
}

// Arrive on the barrier at this shared-memory offset in both CTAs of the pair
// once the preceding MMAs of this thread have completed.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            bar),
        "h"((uint16_t)3)
        : "memory");
}

__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// pdl: as for gemm_kernel (each CTA of the pair copies its B halves of the
// first stages before the dependency wait and its A halves after it).
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm2_kernel(const __grid_constant__ CUtensorMap tma_a, const __grid_constant__ CUtensorMap tma_b,
                 uint16_t *__restrict__ y, int M, int N, int K, int pdl, int b3d) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = (uint32_t)__cvta_generic_to_shared(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    const uint32_t bar0 = base + ST2 * STAGE2_BYTES;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (ST2 + s); };
    auto accf_bar = [&](int a) { return bar0 + 8u * (2 * ST2 + a); };
    auto acce_bar = [&](int a) { return bar0 + 8u * (2 * ST2 + 2 + a); };
    const uint32_t done_bar = bar0 + 8u * (2 * ST2 + 4);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + ST2 * STAGE2_BYTES + 8 * (2 * ST2 + 5));

    pdl_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
    const int tiles_m = (M + 255) / 256, tiles_n = (N + BN - 1) / BN;
    const int ntiles = tiles_m * tiles_n;
    const int nk = (K + BK - 1) / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < ST2; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(accf_bar(a), 1);
            mbar_init(acce_bar(a), 8);  // 4 epilogue warps in each CTA of the pair
        }
        mbar_init(done_bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(&tma_a) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(&tma_b) : "memory");
    }
    if (warp == 1) {
        // One warp of each CTA of the pair allocates collectively.
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         (uint32_t)__cvta_generic_to_shared(tmem_slot)),
                     "r"(TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // both CTAs' barriers exist before any remote signal
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer (both CTAs) ----------------
            uint32_t issued_ph = 0, issued_any = 0;
            int it = 0;
            bool ok = true;
            int pre = 0;  // first-tile stages whose B copies precede the dependency wait
            if (pdl && pair < ntiles) {
                const int m0 = (pair % tiles_m) * 256 + 128 * (int)rank;
                const int n0 = (pair / tiles_m) * BN + 128 * (int)rank;
                pre = nk < ST2 ? nk : ST2;
                for (int kb = 0; kb < pre; ++kb) {  // fresh slots: no empty wait
                    if (rank == 0) mbar_expect_tx(full_bar(kb), 2 * STAGE2_BYTES);
                    const uint32_t lbar = map_to_rank(full_bar(kb), 0);
                    const uint32_t sb = base + kb * STAGE2_BYTES + A2_TILE;
                    load_b_half_pair(sb, &tma_b, n0, kb * BK, lbar, b3d);
                    issued_any |= 1u << kb;
                }
                pdl_wait();
                for (int kb = 0; kb < pre; ++kb)
                    tma_load_2d_pair(base + kb * STAGE2_BYTES, &tma_a, kb * BK, m0, map_to_rank(full_bar(kb), 0));
                it = pre;
            } else if (pdl) {
                pdl_wait();
            }
            for (int t = pair; t < ntiles && ok; t += npairs) {
                const int m0 = (t % tiles_m) * 256 + 128 * (int)rank;
                const int n0 = (t / tiles_m) * BN + 128 * (int)rank;
                for (int kb = (t == pair) ? pre : 0; kb < nk; ++kb, ++it) {
                    const int s = it % ST2;
                    const uint32_t ph = (it / ST2) & 1;
                    if (!mbar_wait(empty_bar(s), ph ^ 1)) {
                        ok = false;
                        break;
                    }
                    if (rank == 0) mbar_expect_tx(full_bar(s), 2 * STAGE2_BYTES);
                    const uint32_t lbar = map_to_rank(full_bar(s), 0);
                    const uint32_t sa = base + s * STAGE2_BYTES;
                    const uint32_t sb = sa + A2_TILE;
                    tma_load_2d_pair(sa, &tma_a, kb * BK, m0, lbar);
                    load_b_half_pair(sb, &tma_b, n0, kb * BK, lbar, b3d);
                    issued_ph = (issued_ph & ~(1u << s)) | (ph << s);
                    issued_any |= 1u << s;
                }
            }
            // The leader's stage barriers count both CTAs' copies: the leader
            // drains them; the final cluster barrier holds the peer until then.
            if (rank == 0)
                for (int s = 0; s < ST2; ++s)
                    if (issued_any & (1u << s)) mbar_wait(full_bar(s), (issued_ph >> s) & 1);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            if (rank == 0) {
                // ---------------- MMA issuer (leader CTA) ----------------
                int it = 0, tc = 0;
                bool ok = true;
                for (int t = pair; t < ntiles && ok; t += npairs, ++tc) {
                    const int acc = tc & 1;
                    const uint32_t aph = (tc >> 1) & 1;
                    if (!mbar_wait(acce_bar(acc), aph ^ 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t dst = tmem + acc * BN;
                    for (int kb = 0; kb < nk; ++kb, ++it) {
                        const int s = it % ST2;
                        const uint32_t ph = (it / ST2) & 1;
                        if (!mbar_wait(full_bar(s), ph)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t sa = base + s * STAGE2_BYTES;
                        const uint32_t sb = sa + A2_TILE;
#pragma unroll
                        for (int ks = 0; ks < BK / 16; ++ks) {
                            const uint64_t ad = smem_desc(sa + ks * 32, 16, 1024);
                            const uint64_t bd = smem_desc(sb + ks * 2048, B_BOX, 1024);
                            mma_f16_pair(dst, ad, bd, (kb | ks) != 0);
                        }
                        mma_commit_pair(empty_bar(s));
                    }
                    if (!ok) break;
                    mma_commit_pair(accf_bar(acc));
                }
                mma_commit_pair(done_bar);
            }
            mbar_wait(done_bar, 0);
        }
    } else {
        // ---------------- epilogue: warps 2..5 of both CTAs ----------------
        const int quad = warp & 3;
        int tc = 0;
        for (int t = pair; t < ntiles; t += npairs, ++tc) {
            const int m0 = (t % tiles_m) * 256 + 128 * (int)rank, n0 = (t / tiles_m) * BN;
            const int acc = tc & 1;
            const uint32_t aph = (tc >> 1) & 1;
            if (!mbar_wait(accf_bar(acc), aph)) break;
            tc_fence_after();
            const int row = m0 + quad * 32 + lane;
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t r[32];
                tmem_ld32(tmem + ((uint32_t)(quad * 32) << 16) + acc * BN + c * 32, r);
                if (c == BN / 32 - 1) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_remote(map_to_rank(acce_bar(acc), 0));
                }
                if (row < M) {
                    uint16_t *dst = y + (size_t)row * N + n0 + c * 32;
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        if (n0 + c * 32 + 8 * v < N) {
                            uint4 o;
                            o.x = pack_half2(r[8 * v + 0], r[8 * v + 1]);
                            o.y = pack_half2(r[8 * v + 2], r[8 * v + 3]);
                            o.z = pack_half2(r[8 * v + 4], r[8 * v + 5]);
                            o.w = pack_half2(r[8 * v + 6], r[8 * v + 7]);
                            *reinterpret_cast<uint4 *>(dst + 8 * v) = o;
                        }
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS));
    }
}

// ---------------------------------------------------------------------------
// w4_gemm: the int4 GEMM with the dequantisation inside the tensor-core
// pipeline, for prefill with few activation rows (M <= 128).  The weight is
// read once as 4-bit codes (0.5625 B per weight for group-64 affine) instead
// of being dequantised into a half scratch (2 B written + 2 B read per
// weight) and then multiplied.
//
// The MMA runs transposed: A = a 128-row weight tile (the MMA's M), held in
// tensor memory; B = the activation tile X (its N = M rounded up to 16,
// K-major in shared memory); D[n][m] = sum_k w[n][k] x[m][k] accumulates in
// tensor memory with one weight row per lane.
//  * Tiles of 128 weight rows, one CTA per SM (G CTAs).  Each CTA takes
//    tiles / G whole tiles (tile i G + b for CTA b); the k steps of the
//    remaining tiles are shared out evenly (a contiguous range of the
//    (tile, step) sequence per CTA, stream-K style), so no SM idles for a
//    partial wave.  A unit (a whole tile, or one tile's part of a CTA's
//    range) walks its 64-k steps from a rotation that differs between
//    tiles, so that CTAs working at the same time read different X tiles
//    from L2.
//  * Codes: a ring of 6 stages of 16 KB (128 rows x 256 k: four 64-k steps
//    per tensor copy, 128-byte rows, 128-byte swizzle).  X and converted
//    weights: a ring of 4 operand stages of two 64-k steps each; a step is
//    an X tile (128 rows x 64 k, K-major, 128-byte swizzle, from L2) and 32
//    tensor-memory columns (64 k of binary16 per lane).  One MMA commit
//    releases a whole operand stage.
//  * Warp 0: one thread issues the code copies (weights are constants: no
//    dependency wait).  Warp 14: one thread issues the X copies (after the
//    dependency wait when launched as a programmatic dependent).
//  * Warps 6-13: converters, two teams of four warps taking alternate
//    operand stages; warp w converts the rows of its tensor-memory lane quarter
//    (w % 4): lane l takes row 32 (w % 4) + l, reads its 64 codes of the
//    step (two 16-byte loads, conflict-free under the swizzle) and writes
//    the 32 binary16 pairs (w[n][k], w[n][k+1]) -- exactly the
//    w4_dequant_f16 value, RNE(scale*q + bias) -- with one tensor-memory
//    store.  Scales and biases are loaded one code stage ahead.
//  * Warp 1: one thread issues tcgen05.mma.kind::f16 with A from tensor
//    memory (M = 128, N = M rounded up to 16, K = 16), four per step and
//    eight per operand stage, then one commit for the stage.
//  * Warps 2-5: epilogue (lane quarter w % 4).  A whole tile: round and
//    store y.  A part of a shared tile: write the fp32 partial tile to the
//    CTA's workspace slot.  For M > 32 the CTA flags it (the call's epoch +
//    1); at the end each CTA waits for the flags of the CTAs it shares a tile
//    with (the launch is cooperative: all resident) and sums its slice of
//    that tile's partials in ascending k; the last CTA to finish advances the
//    epoch.  For M <= 32 the CTA counts its arrival on the tile, and the
//    last to arrive sums the whole tile (nobody waits).
// The binary16 operands are those of f16_gemm on the w4_dequant_f16 scratch;
// only the order of the 64-k steps in the fp32 accumulation differs.
// ---------------------------------------------------------------------------
constexpr int FBN = 128;                              // weight rows per tile
constexpr int QST = 4;                                // operand stages (X tiles + converted weights)
constexpr int QSK = 2;                                // 64-k steps per operand stage
constexpr int QCST = 6;                               // code stages
constexpr int QCK = 4;                                // 64-k steps per code stage (two operand stages)
constexpr int QFX = BM * BK * 2;                      // 16 KB: X, 128 rows x 64 k (one step)
constexpr int QFC = FBN * 128;                        // 16 KB code stage: 128 rows x 32 words
constexpr int Q_TEAM = 4;                             // converter warps per team (one per lane quarter)
constexpr int Q_CONV0 = 6;
constexpr int Q_XWARP = Q_CONV0 + 2 * Q_TEAM;         // 14
constexpr int F_THREADS = (Q_XWARP + 1) * 32;         // 480
constexpr int Q_ACC_COLS = 128;                       // one accumulator: up to 128 activation rows
constexpr int Q_A_COL0 = 2 * Q_ACC_COLS;              // converted weights after the two accumulators
constexpr int F_TMEM_COLS = 512;
constexpr int F_BARS = 2 * QCST + 3 * QST + 5;
constexpr size_t F_SMEM = 1024 + (size_t)QST * QSK * QFX + (size_t)QCST * QFC + 8 * F_BARS + 16;
constexpr int kW4MaxGrid = 256;                       // CTAs per launch (>= the SMs of the GPU)
static_assert(QST >= 2, "converted-weight stage waits rely on at least two stages");
static_assert(QCK == 2 * QSK, "a code stage holds two operand stages");
static_assert(Q_A_COL0 + QST * QSK * 32 <= F_TMEM_COLS, "tensor-memory columns");
static_assert(F_SMEM <= 227 * 1024, "shared memory");

struct W4GemmArgs {
    const uint16_t *sc, *bi;  // scales, biases (null: symmetric codes)
    uint16_t *y;              // [M][N]
    float *part;              // [2 * grid][M][128] fp32 partial tiles (split > 0)
    unsigned *bar;            // [0] CTAs finished, [1] call epoch (zero before the first call)
    unsigned *flags;          // [2 * grid] epoch + 1 once the partial tile of that slot is stored (split 1)
    unsigned *tcnt;           // [remaining tiles] arrivals of a shared tile's CTAs (split 2), zero between calls
    int M, N, K;
    WFmt f;
    int fw;                   // whole tiles per CTA (tile w * grid + b for CTA b)
    int spc;                  // k steps per CTA on the remaining tiles
    int split;                // remaining tiles shared by several CTAs: 0 none; 1 the sharers wait for
                              // each other's flags and each sums a slice; 2 the last to arrive sums it
    int pdl;
    uint32_t idesc;           // instruction descriptor (N = M rounded up to 16)
};

// D[tmem_d] (+)= A[tmem_a] * B[bdesc]: A from tensor memory.
__device__ __forceinline__ void mma_f16_tmem_a(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc, uint32_t idesc,
                                               uint32_t accum) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(tmem_d),
        "r"(tmem_a), "l"(bdesc), "r"(idesc), "r"(accum));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]),
        "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]),
        "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Item it of slice j of c of remaining tile t (shared by CTAs bf .. bf + c
// - 1; an item is 8 columns of one row): the partial sums of its CTAs
// (ascending CTA index = ascending k) added in that order, rounded once and
// stored.  The loads of up to 8 partials are in flight together.
__device__ __forceinline__ void reduce_item(const W4GemmArgs &a, int nk, int G, int rtot, int t, int bf, int c,
                                            int it) {
    const int M = a.M, N = a.N, spc = a.spc, bl = bf + c - 1;
    const int m = it / (FBN / 8), cc = it % (FBN / 8);
    const int n = (a.fw * G + t) * FBN + 8 * cc;
    if (m >= M || n >= N) return;
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    for (int b0 = bf; b0 <= bl; b0 += 8) {
        float4 p0[8], p1[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int b = b0 + q;
            if (b <= bl) {
                const int slot = 2 * b + (min((b + 1) * spc, rtot) <= (t + 1) * nk ? 1 : 0);
                const float *src = a.part + ((size_t)slot * M + m) * FBN + 8 * cc;
                p0[q] = __ldcg(reinterpret_cast<const float4 *>(src));
                p1[q] = __ldcg(reinterpret_cast<const float4 *>(src + 4));
            }
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            if (b0 + q > bl) break;
            acc[0] += p0[q].x; acc[1] += p0[q].y; acc[2] += p0[q].z; acc[3] += p0[q].w;
            acc[4] += p1[q].x; acc[5] += p1[q].y; acc[6] += p1[q].z; acc[7] += p1[q].w;
        }
    }
    uint4 o;
    o.x = pack_half2(__float_as_uint(acc[0]), __float_as_uint(acc[1]));
    o.y = pack_half2(__float_as_uint(acc[2]), __float_as_uint(acc[3]));
    o.z = pack_half2(__float_as_uint(acc[4]), __float_as_uint(acc[5]));
    o.w = pack_half2(__float_as_uint(acc[6]), __float_as_uint(acc[7]));
    *reinterpret_cast<uint4 *>(a.y + (size_t)m * N + n) = o;
}

__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__global__ void __launch_bounds__(F_THREADS, 1)
    w4gemm_kernel(const __grid_constant__ CUtensorMap tma_x, const __grid_constant__ CUtensorMap tma_q,
                  const __grid_constant__ W4GemmArgs a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = (uint32_t)__cvta_generic_to_shared(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    const uint32_t codes0 = base + QST * QSK * QFX;         // code ring
    const uint32_t bar0 = codes0 + QCST * QFC;
    auto code_full = [&](int c) { return bar0 + 8u * c; };                   // codes landed
    auto code_empty = [&](int c) { return bar0 + 8u * (QCST + c); };         // codes read by every converter
    auto x_full = [&](int s) { return bar0 + 8u * (2 * QCST + s); };         // X tile landed
    auto a_full = [&](int s) { return bar0 + 8u * (2 * QCST + QST + s); };   // weights converted
    auto st_empty = [&](int s) { return bar0 + 8u * (2 * QCST + 2 * QST + s); };  // MMAs done with stage s
    auto accf_bar = [&](int x) { return bar0 + 8u * (2 * QCST + 3 * QST + x); };
    auto acce_bar = [&](int x) { return bar0 + 8u * (2 * QCST + 3 * QST + 2 + x); };
    const uint32_t done_bar = bar0 + 8u * (2 * QCST + 3 * QST + 4);
    const size_t tail_off = (size_t)QST * QSK * QFX + (size_t)QCST * QFC + 8 * F_BARS;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + tail_off);
    volatile int *bar_failed = reinterpret_cast<volatile int *>(gbase + tail_off + 4);
    volatile unsigned *epoch_sh = reinterpret_cast<volatile unsigned *>(gbase + tail_off + 8);
    volatile int *last_sh = reinterpret_cast<volatile int *>(gbase + tail_off + 12);

    pdl_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int M = a.M, N = a.N, G = (int)gridDim.x, blk = (int)blockIdx.x;
    const int nk = a.K / BK;
    const int tiles = (N + FBN - 1) / FBN;
    const int rtiles = tiles - a.fw * G;  // tiles shared out by k steps
    const int rtot = rtiles * nk;
    const int l0 = blk * a.spc, l1 = min(l0 + a.spc, rtot);  // this CTA's steps of them
    // Work unit i of this CTA: first its whole tiles (tile i * G + blk, all
    // nk steps), then the pieces of its step range [l0, l1) of the remaining
    // tiles, one per tile it touches (step l is k step l % nk of remaining
    // tile l / nk).  Returns false past the last unit.
    auto unit_range = [&](int i, int &tile, int &kb0, int &kb1) {
        if (i < a.fw) {
            tile = i * G + blk;
            kb0 = 0;
            kb1 = nk;
            return true;
        }
        if (l0 >= l1) return false;
        const int t = l0 / nk + (i - a.fw);
        const int s0 = max(l0, t * nk), s1 = min(l1, (t + 1) * nk);
        if (s0 >= s1) return false;
        tile = a.fw * G + t;
        kb0 = s0 - t * nk;
        kb1 = s1 - t * nk;
        return true;
    };
    // A unit walks its k steps starting at kb0 + rot and wrapping around, rot
    // a multiple of a code stage that differs between tiles: CTAs working on
    // different tiles at the same time then read different X tiles, instead
    // of all of them asking L2 for the same one.
    auto unit_rot = [&](int tile, int kb0, int kb1) {
        const int ns = kb1 - kb0;
        return ns % QCK ? 0 : (int)(((unsigned)tile * 5u) % (unsigned)(ns / QCK)) * QCK;
    };
    auto seq_kb = [](int kb0, int kb1, int rot, int j) {
        int v = j + rot;
        if (v >= kb1 - kb0) v -= kb1 - kb0;
        return kb0 + v;
    };

    if (threadIdx.x == 0) {
        for (int c = 0; c < QCST; ++c) {
            mbar_init(code_full(c), 1);
            mbar_init(code_empty(c), 2 * Q_TEAM);
        }
        for (int s = 0; s < QST; ++s) {
            mbar_init(x_full(s), 1);
            mbar_init(a_full(s), Q_TEAM);
            mbar_init(st_empty(s), 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(accf_bar(x), 1);
            mbar_init(acce_bar(x), 4);
        }
        mbar_init(done_bar, 1);
        *bar_failed = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(&tma_x) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(&tma_q) : "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         (uint32_t)__cvta_generic_to_shared(tmem_slot)),
                     "r"(F_TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- code producer (weights: no dependency wait) ----------------
            uint32_t issued_ph = 0, issued_any = 0;
            int cs = 0;  // code stages issued
            bool ok = true;
            int tile, kb0, kb1;
            for (int u = 0; ok && unit_range(u, tile, kb0, kb1); ++u) {
                const int n0 = tile * FBN;
                const int rot = unit_rot(tile, kb0, kb1);
                for (int j = 0; j < kb1 - kb0; j += QCK, ++cs) {
                    const int c = cs % QCST;
                    const uint32_t ph = (cs / QCST) & 1;
                    if (!mbar_wait(code_empty(c), ph ^ 1)) {
                        ok = false;
                        break;
                    }
                    // Steps k .. k+3 (words 8k ..); past K the copy fills zeros.
                    const int k = seq_kb(kb0, kb1, rot, j);
                    mbar_expect_tx(code_full(c), QFC);
                    tma_load_2d(codes0 + c * QFC, &tma_q, 8 * k, n0, code_full(c));
                    issued_ph = (issued_ph & ~(1u << c)) | (ph << c);
                    issued_any |= 1u << c;
                }
            }
            // Drain: every copy this thread issued has landed before exit.
            for (int c = 0; c < QCST; ++c)
                if (issued_any & (1u << c)) mbar_wait(code_full(c), (issued_ph >> c) & 1);
        }
    } else if (warp == Q_XWARP) {
        if (lane == 0) {
            // ---------------- X producer ----------------
            if (a.pdl) pdl_wait();  // x may be written by the previous kernel
            uint32_t issued_ph = 0, issued_any = 0;
            int g = 0;  // operand stages of this CTA
            bool ok = true;
            int tile, kb0, kb1;
            for (int u = 0; ok && unit_range(u, tile, kb0, kb1); ++u) {
                const int rot = unit_rot(tile, kb0, kb1), ns = kb1 - kb0;
                for (int j = 0; j < ns; j += QSK, ++g) {
                    const int s = g % QST;
                    const uint32_t ph = (g / QST) & 1;
                    if (!mbar_wait(st_empty(s), ph ^ 1)) {
                        ok = false;
                        break;
                    }
                    const int n = min(QSK, ns - j);  // steps of this stage
                    mbar_expect_tx(x_full(s), n * QFX);
                    for (int i = 0; i < n; ++i)
                        tma_load_2d(base + (s * QSK + i) * QFX, &tma_x, seq_kb(kb0, kb1, rot, j + i) * BK, 0,
                                    x_full(s));
                    issued_ph = (issued_ph & ~(1u << s)) | (ph << s);
                    issued_any |= 1u << s;
                }
            }
            for (int s = 0; s < QST; ++s)
                if (issued_any & (1u << s)) mbar_wait(x_full(s), (issued_ph >> s) & 1);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            int g = 0, tc = 0;
            bool ok = true;
            int tile, kb0, kb1;
            for (int u = 0; ok && unit_range(u, tile, kb0, kb1); ++u, ++tc) {
                const int ns = kb1 - kb0;
                const int acc = tc & 1;
                const uint32_t aph = (tc >> 1) & 1;
                if (!mbar_wait(acce_bar(acc), aph ^ 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t dst = tmem + acc * Q_ACC_COLS;
                // Stage s, step i: X at base + (s * QSK + i) * QFX (descriptor
                // address field + that / 16), converted weights at
                // tensor-memory column Q_A_COL0 + 32 (s * QSK + i); each 16-k
                // slice is 32 bytes (+2) or 8 columns further.
                const uint64_t xd0 = smem_desc(base, 16, 1024);
                for (int j = 0; j < ns; j += QSK, ++g) {
                    const int sx = g % QST;
                    const uint32_t ph = (g / QST) & 1;
                    if (!mbar_wait(x_full(sx), ph) || !mbar_wait(a_full(sx), ph)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t bd = xd0 + (uint64_t)(sx * QSK * (QFX >> 4));
                    const uint32_t ta = tmem + Q_A_COL0 + sx * QSK * 32;
                    mma_f16_tmem_a(dst, ta, bd, a.idesc, j != 0 ? 1u : 0u);
                    mma_f16_tmem_a(dst, ta + 8, bd + 2, a.idesc, 1u);
                    mma_f16_tmem_a(dst, ta + 16, bd + 4, a.idesc, 1u);
                    mma_f16_tmem_a(dst, ta + 24, bd + 6, a.idesc, 1u);
                    if (j + 1 < ns) {
                        const uint64_t bd1 = bd + (uint64_t)(QFX >> 4);
                        mma_f16_tmem_a(dst, ta + 32, bd1, a.idesc, 1u);
                        mma_f16_tmem_a(dst, ta + 40, bd1 + 2, a.idesc, 1u);
                        mma_f16_tmem_a(dst, ta + 48, bd1 + 4, a.idesc, 1u);
                        mma_f16_tmem_a(dst, ta + 56, bd1 + 6, a.idesc, 1u);
                    }
                    mma_commit(st_empty(sx));
                }
                if (!ok) break;
                mma_commit(accf_bar(acc));
            }
            mma_commit(done_bar);
            mbar_wait(done_bar, 0);
        }
    } else if (warp >= 2 && warp < Q_CONV0) {
        // ---------------- epilogue: warps 2..5 ----------------
        // Lane l of warp w holds weight row n0 + 32 (w % 4) + l; columns are
        // activation rows.  A unit that covers its whole tile stores y; a
        // piece of a shared tile stores its fp32 partial sums in the slot of
        // this CTA (2 blk for its first unit of the remaining tiles when that
        // is not also its last, 2 blk + 1 for its last) and then flags the
        // slot with the call's epoch + 1.  After an expired wait a warp skips
        // its work but still takes part in the named barriers of every unit.
        const int quad = warp & 3;
        int tc = 0;
        const int ncol = (M + 31) / 32;  // 32-column chunks that hold activation rows
        unsigned ep1 = 0;
        if (a.split == 1 && warp == 2 && lane == 0) {
            pdl_wait();  // the previous call on this workspace has finished
            unsigned e;
            asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(e) : "l"(a.bar + 1) : "memory");
            *epoch_sh = e;
            ep1 = e + 1u;
        }
        bool ok = true;
        int tile, kb0, kb1;
        for (int u = 0; unit_range(u, tile, kb0, kb1); ++u, ++tc) {
            const int n0 = tile * FBN;
            const int acc = tc & 1;
            const uint32_t aph = (tc >> 1) & 1;
            const int n = n0 + quad * 32 + lane;
            if (ok && !mbar_wait(accf_bar(acc), aph)) ok = false;
            if (ok) tc_fence_after();
            const bool whole = kb0 == 0 && kb1 == nk;
            const int t = tile - a.fw * G;  // remaining-tile index (whole == false only there)
            const int slot = 2 * blk + (l1 <= (t + 1) * nk ? 1 : 0);
            for (int c = 0; c < ncol && ok; ++c) {
                uint32_t r[32];
                tmem_ld32(tmem + ((uint32_t)(quad * 32) << 16) + acc * Q_ACC_COLS + c * 32, r);
                if (c == ncol - 1) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(acce_bar(acc));
                }
                if (n >= N) continue;
                const int m0 = c * 32;
                if (whole) {
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (m0 + i < M) a.y[(size_t)(m0 + i) * N + n] = __half_as_ushort(__float2half_rn(__uint_as_float(r[i])));
                } else {
                    float *dst = a.part + (size_t)slot * M * FBN + (n - n0);
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (m0 + i < M) __stcg(dst + (size_t)(m0 + i) * FBN, __uint_as_float(r[i]));
                }
            }
            if (!whole) {
                // The named barrier orders the four warps' stores before the
                // flag or the arrival (the fence is cumulative at gpu scope).
                epi_sync();
                if (a.split == 1) {
                    if (warp == 2 && lane == 0) {
                        __threadfence();
                        asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(a.flags + slot), "r"(ep1) : "memory");
                    }
                } else {
                    // The CTA that brings the tile's last partial sums them
                    // all (no CTA waits) and resets the count for the next call.
                    const int bf = (t * nk) / a.spc, bl = min(G - 1, ((t + 1) * nk - 1) / a.spc);
                    if (warp == 2 && lane == 0) {
                        __threadfence();
                        const unsigned prev = atomicAdd(a.tcnt + t, 1u);
                        const int last = prev == (unsigned)(bl - bf);
                        if (last) a.tcnt[t] = 0u;
                        *last_sh = last;
                    }
                    epi_sync();
                    if (*last_sh && ok) {
                        __threadfence();
                        for (int it = (warp - 2) * 32 + lane; it < M * (FBN / 8); it += 128)
                            reduce_item(a, nk, G, rtot, t, bf, bl - bf + 1, it);
                    }
                    epi_sync();  // every epilogue thread has read the flag before the next unit
                }
            }
        }
    } else if (warp >= Q_CONV0 && warp < Q_XWARP) {
        // ---------------- converters: warps 6..13, two teams ----------------
        const int cw = warp - Q_CONV0;
        const int team = cw / Q_TEAM;
        const int quad = warp & 3;           // tensor-memory lane quarter of this warp
        const int rl = quad * 32 + lane;     // the lane's row within the tile
        const int sw = rl & 7;               // 128-byte swizzle phase of that row
        const bool sym = a.f.sym != 0;
        const __half2 koff = __float2half2_rn(sym ? 1032.f : 1024.f);
        const int ngs = a.f.ngs, gshift = a.f.gs + 5;
        const uint32_t trow = tmem + ((uint32_t)(quad * 32) << 16) + Q_A_COL0;
        // Position of a code stage of this CTA: unit u (rows n0, steps
        // [kb0, kb1) walked from rotation rot), the sequence position j of its
        // first step, and the CTA operand-stage index gs of that step's stage
        // (operand stages pair steps 2i, 2i + 1 of a unit and alternate
        // between the two teams).
        struct CPos {
            int u, n0, kb0, kb1, rot, j, gs;
            bool valid;
        };
        auto cset = [&](CPos &q) {
            int tile;
            q.valid = unit_range(q.u, tile, q.kb0, q.kb1);
            if (q.valid) {
                q.n0 = tile * FBN;
                q.rot = unit_rot(tile, q.kb0, q.kb1);
                q.j = 0;
            }
        };
        auto cstep = [&](CPos &q) {
            const int j1 = q.j + QCK;
            if (j1 < q.kb1 - q.kb0) {
                q.gs += QCK / QSK;
                q.j = j1;
                return;
            }
            q.gs += (q.kb1 - q.kb0 - q.j + QSK - 1) / QSK;
            ++q.u;
            cset(q);
        };
        // Scales (and biases) of the two 32-k halves of this team's steps of
        // the code stage at q, as binary16 bit patterns (loaded one code
        // stage ahead, so that no step waits for them).
        auto load_sb = [&](const CPos &q, uint32_t (&sv)[QCK], uint32_t (&bv)[QCK]) {
            const int row = min(q.n0 + rl, N - 1);  // rows past N: any valid scales (results unused)
            const uint16_t *srow = a.sc + (size_t)row * ngs;
            const uint16_t *brow = a.bi + (size_t)row * ngs;
#pragma unroll
            for (int j = 0; j < QCK; ++j) {
                sv[j] = bv[j] = 0u;
                if (q.j + j >= q.kb1 - q.kb0 || ((q.gs + j / QSK) & 1) != team) continue;
                const int kb = seq_kb(q.kb0, q.kb1, q.rot, q.j + j);
                const int g0 = (kb * BK) >> gshift, g1 = (kb * BK + 32) >> gshift;
                sv[j] = (uint32_t)ld_nc_u16(srow + g0) | ((uint32_t)ld_nc_u16(srow + g1) << 16);
                if (!sym) bv[j] = (uint32_t)ld_nc_u16(brow + g0) | ((uint32_t)ld_nc_u16(brow + g1) << 16);
            }
        };
        CPos pf;
        pf.u = 0;
        pf.gs = 0;
        cset(pf);
        uint32_t nxs[QCK], nxb[QCK];
        if (pf.valid) load_sb(pf, nxs, nxb);
        bool ok = true;
        int cs = 0;  // code stages
        while (pf.valid && ok) {
            const CPos cur = pf;
            uint32_t cus[QCK], cub[QCK];
#pragma unroll
            for (int j = 0; j < QCK; ++j) {
                cus[j] = nxs[j];
                cub[j] = nxb[j];
            }
            cstep(pf);
            if (pf.valid) load_sb(pf, nxs, nxb);
            const int c = cs % QCST;
            if (!mbar_wait(code_full(c), (cs / QCST) & 1)) {
                ok = false;
                break;
            }
            const uint32_t crow = codes0 + c * QFC + rl * 128;
            const int ns = cur.kb1 - cur.kb0;
#pragma unroll
            for (int q = 0; q < QCK / QSK; ++q) {
                const int g = cur.gs + q;            // operand stage of steps j, j + 1
                const int jq = cur.j + QSK * q;
                if (jq >= ns) break;
                if ((g & 1) != team) continue;      // the other team's stage
                const int sa = g % QST;
                // The stage is free once the MMAs of its previous use (stage
                // g - QST) are done; this team's previous stage (g - 2)
                // waited for stage g - 2 - QST, so with QST >= 2 every earlier
                // phase of the barrier is complete and the parity cannot alias.
                if (!mbar_wait(st_empty(sa), ((g / QST) & 1) ^ 1)) {
                    ok = false;
                    break;
                }
#pragma unroll
                for (int i = 0; i < QSK; ++i) {
                    const int j = QSK * q + i;        // step within the code stage
                    if (jq + i >= ns) break;
                    const uint4 qa = lds128(crow + (((2 * j) ^ sw) << 4));
                    const uint4 qb = lds128(crow + (((2 * j + 1) ^ sw) << 4));
                    uint32_t out[32];
                    const uint32_t wd[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
#pragma unroll
                    for (int w = 0; w < 8; ++w) {
                        // Scale and bias of the word's 32-k half, in both halves.
                        const uint32_t sv = w < 4 ? __byte_perm(cus[j], 0, 0x1010) : __byte_perm(cus[j], 0, 0x3232);
                        const uint32_t bv = w < 4 ? __byte_perm(cub[j], 0, 0x1010) : __byte_perm(cub[j], 0, 0x3232);
                        const __half2 s2 = *reinterpret_cast<const __half2 *>(&sv);
                        const __half2 b2 = *reinterpret_cast<const __half2 *>(&bv);
                        const uint32_t x = wd[w], x4 = x >> 4;
                        // Codes (2e, 2e + 1) of the word into the two halves:
                        // bytes e of x and of x >> 4, low nibbles.
                        const uint32_t p[4] = {__byte_perm(x, x4, 0x5410), __byte_perm(x, x4, 0x6521),
                                               __byte_perm(x, x4, 0x7632), __byte_perm(x, x4, 0x7733)};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const uint32_t qv = (p[e] & 0x000F000Fu) | 0x64006400u;  // 1024 + q
                            const __half2 q2 = __hsub2(*reinterpret_cast<const __half2 *>(&qv), koff);
                            const __half2 w2 = sym ? __hmul2(q2, s2) : __hfma2(q2, s2, b2);  // one rounding
                            out[4 * w + e] = *reinterpret_cast<const uint32_t *>(&w2);
                        }
                    }
                    tmem_st32(trow + (sa * QSK + i) * 32, out);
                }
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(a_full(sa));
            }
            if (!ok) break;
            // Every converter warp reads every code stage (its own steps);
            // its reads are ordered before the next tensor copy into the slot.
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(code_empty(c));
            ++cs;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(F_TMEM_COLS));
    }
    if (a.split != 1) return;
    // The shared tiles this CTA touched (at most two: the first and last tile
    // of its step range; the ones between are whole): wait until every CTA
    // that shares one of them has flagged its partial tile (the launch is
    // cooperative, so they are all resident; bounded), then sum slice
    // blk - bf of each, both tiles' items in one pass.
    const unsigned want = *epoch_sh + 1u;
    int st_t[2], st_bf[2], st_c[2], nst = 0;
    if (l0 < l1) {
        const int tf = l0 / nk, tl = (l1 - 1) / nk;
        for (int t = tf; t <= tl; t += (tl > tf ? tl - tf : 1)) {
            const int bf = (t * nk) / a.spc, bl = min(G - 1, ((t + 1) * nk - 1) / a.spc);
            if (bf == bl) continue;
            st_t[nst] = t;
            st_bf[nst] = bf;
            st_c[nst] = bl - bf + 1;
            ++nst;
        }
    }
    if (nst > 0) {
        const int cw = st_c[0] + (nst > 1 ? st_c[1] : 0);
        for (int i = threadIdx.x; i < cw; i += blockDim.x) {
            const int k = i < st_c[0] ? 0 : 1;
            const int t = st_t[k], b = st_bf[k] + (k ? i - st_c[0] : i);
            const int slot = 2 * b + (min((b + 1) * a.spc, rtot) <= (t + 1) * nk ? 1 : 0);
            const uint64_t t0 = global_ns();
            while (ld_acquire_u32(a.flags + slot) != want) {
                if (*bar_failed) break;
                if (global_ns() - t0 > kWaitNs) {
                    atomicExch(&g_wait_expired, 1);
                    *bar_failed = 1;
                    break;
                }
            }
        }
        __syncthreads();
        if (!*bar_failed) {
            // Slice j of c of a tile: the contiguous items [j len, (j + 1) len)
            // of its M x 16 (len = ceil(M x 16 / c)), so that neighbouring
            // threads read neighbouring 32-byte chunks.
            const int items = a.M * (FBN / 8);
            int lo[2] = {0, 0}, cnt[2] = {0, 0};
            for (int k = 0; k < nst; ++k) {
                const int len = (items + st_c[k] - 1) / st_c[k];
                lo[k] = (blk - st_bf[k]) * len;
                cnt[k] = max(0, min(items, lo[k] + len) - lo[k]);
            }
            for (int i = threadIdx.x; i < cnt[0] + cnt[1]; i += blockDim.x) {
                const int k = i < cnt[0] ? 0 : 1;
                reduce_item(a, nk, G, rtot, st_t[k], st_bf[k], st_c[k], lo[k] + (k ? i - cnt[0] : i));
            }
        }
    }
    // The last CTA to finish advances the epoch for the next call.
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(a.bar, 1u) == (unsigned)G - 1u) {
            a.bar[0] = 0u;
            __threadfence();
            asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(a.bar + 1), "r"(want) : "memory");
        }
    }
}

bool make_map(CUtensorMap *m, const void *ptr, uint64_t inner, uint64_t outer, uint32_t box_inner,
              uint32_t box_outer) {
    return make_map_2d(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, ptr, inner, outer, inner * 2, box_inner, box_outer,
                       CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace
}  // namespace w4a16

using namespace w4a16;

static int gemm_impl(const uint16_t *x16, const uint16_t *w16, uint16_t *y, int M, int N, int K, unsigned flags,
                     void *stream) {
    if (!x16 || !w16 || !y) return W4_ERR_NULL;
    if (M < 1 || N < 8 || K < 8 || N % 8 != 0 || K % 8 != 0) return W4_ERR_SHAPE;
    if (!aligned16(x16) || !aligned16(w16) || !aligned16(y)) return W4_ERR_ALIGN;
    if (device_cc() != 103) return W4_ERR_DEVICE;
    CUtensorMap ta, tb;
    if (!make_map(&ta, x16, (uint64_t)K, (uint64_t)M, BK, BM)) return W4_ERR_DEVICE;
    if (!make_map(&tb, w16, (uint64_t)N, (uint64_t)K, 64, BK)) return W4_ERR_DEVICE;
    // The pair kernel loads 128-row A boxes (one per CTA) and the same B boxes.
    CUtensorMap ta2 = ta, tb2 = tb;
    // For N a multiple of 64, W16 is also viewed as [N / 64][K][64] so that
    // one copy brings a tile's boxes (BN / 64 of them; two per CTA of a pair).
    const int b3d = (N % 64 == 0) ? 1 : 0;
    if (b3d) {
        if (!make_map_3d(&tb, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, w16, 64, (uint64_t)K, (uint64_t)N / 64, (uint64_t)N * 2,
                         128, 64, BK, BN / 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !make_map_3d(&tb2, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, w16, 64, (uint64_t)K, (uint64_t)N / 64,
                         (uint64_t)N * 2, 128, 64, BK, 2, CU_TENSOR_MAP_SWIZZLE_128B))
            return W4_ERR_DEVICE;
    }
    if (!set_smem_once(reinterpret_cast<const void *>(gemm_kernel), (int)SMEM_BYTES)) return W4_ERR_LAUNCH;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (M > BM) {
        // CTA pairs: 256 x 256 tiles, half the operand traffic per SM.
        if (!set_smem_once(reinterpret_cast<const void *>(gemm2_kernel), (int)SMEM2_BYTES)) return W4_ERR_LAUNCH;
        const int tiles = ((M + 255) / 256) * ((N + BN - 1) / BN);
        int pairs = sm_count() / 2;
        if (pairs > tiles) pairs = tiles;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * pairs, 1, 1);
        cfg.blockDim = dim3(NUM_THREADS, 1, 1);
        cfg.dynamicSmemBytes = SMEM2_BYTES;
        cfg.stream = st;
        const int pdl = (flags & W4A16_OVERLAP_PREVIOUS) ? 1 : 0;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = pdl ? 2 : 1;
        const cudaError_t e = cudaLaunchKernelEx(&cfg, gemm2_kernel, ta2, tb2, y, M, N, K, pdl, b3d);
        return e == cudaSuccess ? W4A16_OK : W4_ERR_LAUNCH;
    }
    const int tiles = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
    int grid = sm_count();
    if (grid > tiles) grid = tiles;
    const int pdl = (flags & W4A16_OVERLAP_PREVIOUS) ? 1 : 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, gemm_kernel, ta, tb, y, M, N, K, pdl, b3d);
    return e == cudaSuccess ? W4A16_OK : W4_ERR_LAUNCH;
}

extern "C" int f16_gemm(const uint16_t *x16, const uint16_t *w16, uint16_t *y, int M, int N, int K,
                        void *stream) {
    return gemm_impl(x16, w16, y, M, N, K, 0u, stream);
}

extern "C" int f16_gemm_ex(const uint16_t *x16, const uint16_t *w16, uint16_t *y, int M, int N, int K,
                           unsigned flags, void *stream) {
    if (flags & ~(unsigned)W4A16_OVERLAP_PREVIOUS) return W4_ERR_SHAPE;
    return gemm_impl(x16, w16, y, M, N, K, flags, stream);
}

// ---------------------------------------------------------------------------
// w4_gemm host side.
// ---------------------------------------------------------------------------
namespace w4a16 {
namespace {

// Work split of w4_gemm over G CTAs (one per SM): fw = tiles / G whole tiles
// per CTA, then the remaining tiles, whose k steps are shared out evenly
// (spc per CTA, at least 8: two code stages) when that saves more than 14
// steps per CTA: a shared tile costs its CTAs about 5 µs more at the end
// (partial stores, the wait for or the count of the other sharers, the sum)
// against about 0.35 µs per 64-k step.  Otherwise each remaining tile goes
// whole to one CTA (spc = nk).  Fewer sharers per tile than one per CTA
// (spc of at least 8) measured faster for the 32-step tiles (fewer partial
// tiles, fewer CTAs reading activation tiles from L2 at once; GB300, M = 16
// ... 128).  A tile touched by several CTAs gets their fp32 partial sums
// added at the end.
struct W4Split {
    int grid, fw, spc, split;
};

W4Split w4gemm_split(int N, int K, int sms) {
    W4Split w;
    const int tiles = (N + FBN - 1) / FBN, nk = K / BK;
    const int G0 = sms < kW4MaxGrid ? sms : kW4MaxGrid;
    w.fw = tiles / G0;
    const int rtiles = tiles - w.fw * G0;
    const int rtot = rtiles * nk;
    w.spc = rtot > 0 ? (rtot + G0 - 1) / G0 : 1;
    const int floor_steps = nk < 2 * QCK ? nk : 2 * QCK;
    if (rtot > 0 && w.spc < floor_steps) w.spc = floor_steps;
    if (rtot > 0 && nk - w.spc <= 14) w.spc = nk;  // whole tiles only
    w.grid = w.fw > 0 ? G0 : (rtot + w.spc - 1) / w.spc;
    w.split = 0;
    for (int t = 0; t < rtiles && !w.split; ++t) {
        const int bf = (t * nk) / w.spc, bl = ((t + 1) * nk - 1) / w.spc;
        if (bf != bl) w.split = 1;
    }
    return w;
}

// Workspace: 256 bytes of counters (CTAs finished, call epoch), one flag per
// partial-tile slot (2 kW4MaxGrid words), one arrival counter per remaining
// tile (kW4MaxGrid words), then two fp32 partial tiles (M x 128) per CTA for
// at most min(kW4MaxGrid, k steps in all) CTAs.
constexpr size_t kW4FlagsOff = 256, kW4CntOff = kW4FlagsOff + 2 * kW4MaxGrid * 4,
                 kW4PartOff = kW4CntOff + kW4MaxGrid * 4;
size_t w4gemm_workspace_need(int M, int N, int K) {
    const long long steps = (long long)((N + FBN - 1) / FBN) * (K / BK);
    const long long grid = steps < kW4MaxGrid ? steps : kW4MaxGrid;
    return kW4PartOff + (size_t)(2 * grid) * (size_t)M * FBN * 4;
}

bool w4gemm_shape_ok(int M, int N, int K) {
    return M >= 1 && M <= BM && N >= 8 && N % 8 == 0 && K >= BK && K % BK == 0;
}

int w4gemm_impl(const uint16_t *x, const uint32_t *qweight, const uint16_t *scales, const uint16_t *biases,
                uint16_t *y, int M, int N, int K, int group, void *workspace, size_t workspace_bytes, unsigned flags,
                void *stream) {
    if (!x || !qweight || !scales || !y) return W4_ERR_NULL;
    if (flags & ~(unsigned)W4A16_OVERLAP_PREVIOUS) return W4_ERR_SHAPE;
    if (!w4gemm_shape_ok(M, N, K)) return W4_ERR_SHAPE;
    WFmt f;
    if (!make_fmt(f, K, group, biases == nullptr)) return W4_ERR_GROUP;
    const size_t need = w4gemm_workspace_need(M, N, K);
    if (!workspace || workspace_bytes < need) return W4_ERR_WORKSPACE;
    if (!aligned16(x) || !aligned16(qweight) || !aligned16(scales) || (biases && !aligned16(biases)) ||
        !aligned16(y) || !aligned16(workspace))
        return W4_ERR_ALIGN;
    if (device_cc() != 103) return W4_ERR_DEVICE;
    CUtensorMap tx, tq;
    if (!make_map(&tx, x, (uint64_t)K, (uint64_t)M, BK, BM)) return W4_ERR_DEVICE;
    // Codes: 128 rows x 32 words (four 64-k steps) per copy, 128-byte swizzle.
    if (!make_map_2d(&tq, CU_TENSOR_MAP_DATA_TYPE_UINT32, qweight, (uint64_t)K / 8, (uint64_t)N, (uint64_t)K / 2,
                     32, FBN, CU_TENSOR_MAP_SWIZZLE_128B))
        return W4_ERR_DEVICE;
    if (!set_smem_once(reinterpret_cast<const void *>(w4gemm_kernel), (int)F_SMEM)) return W4_ERR_LAUNCH;
    const int sms = sm_count();
    W4GemmArgs a;
    a.sc = scales;
    a.bi = biases;
    a.y = y;
    a.bar = reinterpret_cast<unsigned *>(workspace);
    a.flags = reinterpret_cast<unsigned *>(reinterpret_cast<uint8_t *>(workspace) + kW4FlagsOff);
    a.tcnt = reinterpret_cast<unsigned *>(reinterpret_cast<uint8_t *>(workspace) + kW4CntOff);
    a.part = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(workspace) + kW4PartOff);
    a.M = M;
    a.N = N;
    a.K = K;
    a.f = f;
    const W4Split w = w4gemm_split(N, K, sms);
    a.fw = w.fw;
    a.spc = w.spc;
    // Small partial tiles (M <= 32) are summed by the last sharer to arrive;
    // larger ones in slices by all sharers after they wait for each other.
    a.split = w.split ? (M <= 32 ? 2 : 1) : 0;
    a.pdl = (flags & W4A16_OVERLAP_PREVIOUS) ? 1 : 0;
    // kind::f16, fp32 accumulate, A (weights, tensor memory) and B (X) binary16
    // and K-major, N = M rounded up to 16, M = 128 weight rows.
    const uint32_t nmma = (uint32_t)((M + 15) / 16 * 16);
    a.idesc = (1u << 4) | ((nmma >> 3) << 17) | ((uint32_t)(FBN >> 4) << 24);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)w.grid, 1, 1);
    cfg.blockDim = dim3(F_THREADS, 1, 1);
    cfg.dynamicSmemBytes = F_SMEM;
    cfg.stream = reinterpret_cast<cudaStream_t>(stream);
    // CTAs that wait for each other (split 1) must all be resident: a
    // cooperative launch (one CTA per SM fits: grid <= SMs).
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (a.split == 1) {
        attr[na].id = cudaLaunchAttributeCooperative;
        attr[na].val.cooperative = 1;
        ++na;
    }
    if (a.pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, w4gemm_kernel, tx, tq, a);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return W4_ERR_LAUNCH;
    }
    return W4A16_OK;
}

}  // namespace
}  // namespace w4a16

extern "C" size_t w4_gemm_workspace_bytes(int M, int N, int K) {
    if (!w4gemm_shape_ok(M, N, K)) return 0;
    return w4gemm_workspace_need(M, N, K);
}

extern "C" int w4_gemm(const uint16_t *x, const uint32_t *qweight, const uint16_t *scales, const uint16_t *biases,
                       uint16_t *y, int M, int N, int K, int group, void *workspace, size_t workspace_bytes,
                       void *stream) {
    return w4gemm_impl(x, qweight, scales, biases, y, M, N, K, group, workspace, workspace_bytes, 0u, stream);
}

extern "C" int w4_gemm_ex(const uint16_t *x, const uint32_t *qweight, const uint16_t *scales,
                          const uint16_t *biases, uint16_t *y, int M, int N, int K, int group, void *workspace,
                          size_t workspace_bytes, unsigned flags, void *stream) {
    return w4gemm_impl(x, qweight, scales, biases, y, M, N, K, group, workspace, workspace_bytes, flags, stream);
}

namespace w4a16 {
int gemv_wait_flag();     // gemv.cu
int dequant_wait_flag();  // dequant.cu

// Reads and clears this translation unit's expired-wait record.
static int gemm_wait_flag() {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_wait_expired, sizeof(int)) != cudaSuccess) return -1;
    if (v) {
        const int zero = 0;
        cudaMemcpyToSymbol(g_wait_expired, &zero, sizeof(int));
    }
    return v;
}
}  // namespace w4a16

extern "C" int w4a16_device_status(void) {
    if (cudaDeviceSynchronize() != cudaSuccess) return W4_ERR_LAUNCH;
    const int a = gemm_wait_flag(), b = gemv_wait_flag(), c = dequant_wait_flag();
    if (a < 0 || b < 0 || c < 0) return W4_ERR_LAUNCH;
    return (a || b || c) ? W4_ERR_TIMEOUT : W4A16_OK;
}

extern "C" const char *w4a16_status_string(int status) {
    switch (status) {
        case W4A16_OK: return "ok";
        case W4_ERR_NULL: return "null pointer";
        case W4_ERR_SHAPE: return "unsupported shape";
        case W4_ERR_ALIGN: return "pointer or stride not 16-byte aligned";
        case W4_ERR_GROUP: return "group must be a power of two in 32..K that divides K";
        case W4_ERR_LAUNCH: return "CUDA launch error";
        case W4_ERR_WORKSPACE: return "workspace missing or too small";
        case W4_ERR_DEVICE: return "unsupported device (needs sm_103) or missing driver entry point";
        case W4_ERR_TIMEOUT: return "a device-side bounded wait expired";
        default: return "unknown status";
    }
}
