// Shared helpers of the W4A16 CUDA library (sm_103a).
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/w4a16.h"

namespace w4a16 {

// The kernels step along K in blocks of 64 codes (8 words per row); the
// quantisation group is a runtime parameter described by WFmt.
constexpr int kGroup = 64;         // k per code block
constexpr int kWordsPerGroup = 8;  // 64 four-bit codes = 8 words

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Scale layout of a quantised weight: ngs scale (and bias) entries per row
// (K / group); gs = log2(group / 32), so group = 32 << gs; sym: the weight
// has no biases and w = scale * (q - 8) (symmetric codes).
struct WFmt {
    int ngs, gs, sym;
};

// Kernel variants by scale layout: group-64 affine (the workloads' format),
// symmetric group 128, any other group of 64 or more (runtime layout), and
// group 32 (two quantisation groups per 64-k block).
enum : int { kFmtG64 = 0, kFmtAny = 1, kFmtG32 = 2, kFmtS128 = 3 };

inline int fmt_class(const WFmt &f) {
    if (f.gs == 0) return kFmtG32;
    if (f.gs == 1 && !f.sym) return kFmtG64;
    if (f.gs == 2 && f.sym) return kFmtS128;
    return kFmtAny;
}

// Host check of a (K, group) pair: group a power of two with
// 32 <= group <= K and K % group == 0.  Fills f; false if unsupported.
inline bool make_fmt(WFmt &f, int K, int group, bool sym) {
    if (group < 32 || group > K || (group & (group - 1)) != 0 || K % group != 0) return false;
    int gs = 0;
    while ((32 << gs) < group) ++gs;
    f.ngs = K / group;
    f.gs = gs;
    f.sym = sym ? 1 : 0;
    return true;
}

inline int launch_status() {
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? W4A16_OK : W4_ERR_LAUNCH;
}

// Raise a kernel's dynamic shared-memory limit to `bytes` on the current
// device, once per (kernel, device, size) and thread-safe, so that launches
// captured into CUDA graphs make no attribute calls.  False if the runtime
// refuses (its error is cleared).
inline bool set_smem_once(const void *kern, int bytes) {
    struct Entry {
        const void *kern;
        int dev, bytes;
    };
    static std::mutex mu;
    static Entry done[64];
    static int n = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n; ++i)
        if (done[i].kern == kern && done[i].dev == dev && done[i].bytes >= bytes) return true;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (n < 64) done[n++] = Entry{kern, dev, bytes};
    return true;
}

// Number of SMs of the current device (cached per device).
int sm_count();
// Compute capability major*10+minor of the current device (cached per device).
int device_cc();

// ---- device helpers ----

__device__ __forceinline__ uint32_t ld_nc_u32(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.b32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ uint2 ld_nc_u64(const uint32_t *p) {
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.b32 {%0, %1}, [%2];"
                 : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

__device__ __forceinline__ uint16_t ld_nc_u16(const uint16_t *p) {
    uint16_t v;
    asm volatile("ld.global.nc.b16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ float h2f(uint16_t h) { return __half2float(__ushort_as_half(h)); }

// 16-byte shared-memory load at a shared-window address.
__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}

// D(16x8, fp32) += A(16x16, fp16, row) * B(16x8, fp16, col).
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}


// ---- bounded waits, mbarriers, bulk / tensor copies ----

// Set by a kernel of this translation unit when a bounded wait expires
// (one copy per translation unit; read by w4a16_device_status).
static __device__ int g_wait_expired = 0;

constexpr unsigned long long kWaitNs = 2000000000ull;  // 2 s per wait
constexpr uint32_t kMaxSpins = 1u << 26;

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase of parity `parity`.  `abort` (shared memory, may
// be null) is raised by the first wait that expires and makes every later
// wait of the CTA give up at once, so the CTA can still reach its barriers
// and exit.
static __device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, volatile int *abort) {
    const uint64_t t0 = global_ns();
    for (uint32_t spin = 0; spin < kMaxSpins; ++spin) {
        if (mbar_try(bar, parity)) return true;
        if ((spin & 63) == 63) {
            if (abort && *abort) return false;
            if (global_ns() - t0 > kWaitNs) break;
        }
    }
    atomicExch(&g_wait_expired, 1);
    if (abort) *abort = 1;
    return false;
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort = nullptr) {
    return mbar_try(bar, parity) || mbar_wait_slow(bar, parity, abort);
}

// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA / bulk copy) accesses of the same bytes (e.g. a TMA store
// of a tile the threads just wrote).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

// 2-D tensor copy global -> shared, completion counted on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int c0, int c1, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
            "r"(dst),
        "l"(map), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

// 3-D tensor copy global -> shared, completion counted on `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int c0, int c1, int c2,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::
            "r"(dst),
        "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}

// 2-D tensor copy shared -> global, tracked by the issuing thread's bulk
// async-group (commit with bulk_commit_group, wait with bulk_wait_*).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, uint32_t src, int c0, int c1) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(map), "r"(src),
                 "r"(c0), "r"(c1)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Until at most N of this thread's committed groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Until at most N of this thread's committed groups are incomplete.
template <int N>
__device__ __forceinline__ void bulk_wait_group() {
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// Contiguous bulk copy global -> shared (16-byte aligned, size multiple of 16).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// Programmatic dependent launch: let the next kernel on the stream start its
// prologue now; wait until the previous kernel's results are visible.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---- host: tensor maps through the driver entry point (no libcuda link) ----

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// Row-major 2-D tensor [outer][inner] with `row_bytes` between rows.
inline bool make_map_2d(CUtensorMap *m, CUtensorMapDataType dt, const void *ptr, uint64_t inner, uint64_t outer,
                        uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, dt, 2, const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D tensor with dims {d0, d1, d2} (d0 innermost, contiguous) and byte
// strides s1, s2 for dims 1 and 2 (any order of magnitude).
inline bool make_map_3d(CUtensorMap *m, CUtensorMapDataType dt, const void *ptr, uint64_t d0, uint64_t d1,
                        uint64_t d2, uint64_t s1, uint64_t s2, uint32_t b0, uint32_t b1, uint32_t b2,
                        CUtensorMapSwizzle sw) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {s1, s2};
    const cuuint32_t box[3] = {b0, b1, b2};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, dt, 3, const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace w4a16
