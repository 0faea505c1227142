// Decode-side kernels: the W4A16 multi-row GEMV (w4_gemv) and the LM-head
// GEMV fused with greedy / top-k token selection (lm_head_argmax_topk).
//
// "The inference engine - Mojo 1.0 on Metal", "Crossing Mojo 1.0": the decode
// GEMV is weight-streaming bound; each worker owns several output rows and
// keeps independent weight streams in flight, and token selection runs on the
// device so no logits vector is downloaded.
//
// Design (sm_103a):
//  * A warp owns a tile of 16 output rows.  Lane (g, t) = (lane/4, lane%4)
//    streams rows g and g+8 of the tile: for every group of 64 codes it loads
//    words 2t and 2t+1 of each row (8 bytes per row per group; the four lanes
//    of a row cover the group's 32 contiguous bytes).
//  * Codes are unpacked in registers straight into the A operand of an
//    m16n8k16 tensor-core MMA: (word >> 4j) & 0x000F000F places codes j and
//    j+4 in the two halves of a 32-bit register as binary16 subnormals
//    q * 2^-24, which are exact.  The B operand holds the activations of up
//    to 8 (or 16) rows, pre-arranged in shared memory in fragment order so
//    that the k of each A element matches.  Four MMAs cover one group with
//    exact products and fp32 accumulation.
//  * The affine dequantisation is folded per group: with P = sum_{k in g} q x
//    and X = sum_{k in g} x,  sum_k w x = scale * P + bias * X.  X is
//    computed once per CTA; the fp32 accumulators get acc_s += scale * (P *
//    2^-24) and acc_b += bias * X, and y = 2^24 * acc_s + acc_b.
//  * K is split across the warps of a CTA (partials reduced in shared memory
//    in fixed order) and, for matrices with few row tiles, across the CTAs of
//    a thread-block cluster (partials reduced through distributed shared
//    memory by cluster rank 0, fixed order).  Results are deterministic.
#include <cooperative_groups.h>

#include <mutex>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace w4a16 {

int sm_count() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
    if (cache[dev] == 0) {
        int v = 0;
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        cache[dev] = v > 0 ? v : 1;
    }
    return cache[dev];
}

int device_cc() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (cache[dev] == 0) {
        int maj = 0, mnr = 0;
        cudaDeviceGetAttribute(&maj, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&mnr, cudaDevAttrComputeCapabilityMinor, dev);
        cache[dev] = maj * 10 + mnr;
    }
    return cache[dev];
}

namespace {

constexpr int kTileRows = 16;  // output rows per MMA tile
constexpr int kUnroll = 4;     // groups per load batch (two batches in flight)
constexpr uint32_t kNibPair = 0x000F000Fu;
constexpr float kTwo24 = 16777216.0f;

// ---------------------------------------------------------------------------
// Activation staging.  For local group gl, fragment half h (MMAs j = 2h and
// 2h+1), activation row c and lane quad t, four words are stored at
//   xf[(((gl*2 + h)*M + c)*4 + t)*4 ...]  =  {b0(2h), b1(2h), b0(2h+1), b1(2h+1)}
// with b0(j) = (x[c][k+j], x[c][k+j+4]), b1(j) = (x[c][k+8+j], x[c][k+12+j]),
// k = 64G + 16t.  xsum[gl*M + c] = sum of the group's 64 activations (fp32).
// ---------------------------------------------------------------------------
__device__ void stage_activations(const uint16_t *__restrict__ x, int M, int K, int g0, int ngl,
                                  uint32_t *xf, float *xsum) {
    const int items = ngl * M * 4;
    for (int base = 0; base < items; base += blockDim.x) {
        const int it = base + threadIdx.x;
        float part = 0.f;
        if (it < items) {
            const int t = it & 3;
            const int c = (it >> 2) % M;
            const int gl = (it >> 2) / M;
            const uint4 *src =
                reinterpret_cast<const uint4 *>(x + (size_t)c * K + (size_t)(g0 + gl) * kGroup + 16 * t);
            const uint4 lo = __ldg(src), hi = __ldg(src + 1);
            uint4 f0, f1;
            f0.x = __byte_perm(lo.x, lo.z, 0x5410);  // (x0, x4)
            f0.y = __byte_perm(hi.x, hi.z, 0x5410);  // (x8, x12)
            f0.z = __byte_perm(lo.x, lo.z, 0x7632);  // (x1, x5)
            f0.w = __byte_perm(hi.x, hi.z, 0x7632);  // (x9, x13)
            f1.x = __byte_perm(lo.y, lo.w, 0x5410);  // (x2, x6)
            f1.y = __byte_perm(hi.y, hi.w, 0x5410);  // (x10, x14)
            f1.z = __byte_perm(lo.y, lo.w, 0x7632);  // (x3, x7)
            f1.w = __byte_perm(hi.y, hi.w, 0x7632);  // (x11, x15)
            reinterpret_cast<uint4 *>(xf)[((gl * 2 + 0) * M + c) * 4 + t] = f0;
            reinterpret_cast<uint4 *>(xf)[((gl * 2 + 1) * M + c) * 4 + t] = f1;
            const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                part += h2f((uint16_t)(w[i] & 0xFFFFu));
                part += h2f((uint16_t)(w[i] >> 16));
            }
        }
        part += __shfl_xor_sync(0xffffffffu, part, 1);
        part += __shfl_xor_sync(0xffffffffu, part, 2);
        if (it < items && (it & 3) == 0) xsum[it >> 2] = part;
    }
}

template <int NT>
struct Acc {
    float s[NT][4];
    float b[NT][4];
    __device__ __forceinline__ void zero() {
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int i = 0; i < 4; ++i) s[n][i] = b[n][i] = 0.f;
    }
};

// Weight and scale registers of one group for one lane.
struct GroupRegs {
    uint2 wa, wb;       // words 2t, 2t+1 of rows g and g+8
    uint16_t sa, sb;    // scales of rows g, g+8
    uint16_t ba, bb;    // biases of rows g, g+8
};

struct RowPtrs {
    const uint32_t *qa, *qb;   // qweight rows g, g+8 (offset by 2t words)
    const uint16_t *sa, *sb;   // scale rows
    const uint16_t *ba, *bb;   // bias rows
};

__device__ __forceinline__ void load_group(GroupRegs &r, const RowPtrs &p, int G) {
    r.wa = ld_nc_u64(p.qa + (size_t)G * kWordsPerGroup);
    r.wb = ld_nc_u64(p.qb + (size_t)G * kWordsPerGroup);
    r.sa = ld_nc_u16(p.sa + G);
    r.sb = ld_nc_u16(p.sb + G);
    r.ba = ld_nc_u16(p.ba + G);
    r.bb = ld_nc_u16(p.bb + G);
}

// One group of 64 k for the warp's 16-row tile: 4 MMAs per activation tile.
template <int NT>
__device__ __forceinline__ void group_step(Acc<NT> &acc, const GroupRegs &r, const uint32_t *xf,
                                           const float *xsum, int gl, int M, int lg, int lt) {
    uint32_t a0[4], a1[4], a2[4], a3[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        a0[j] = (r.wa.x >> (4 * j)) & kNibPair;  // row g,   cols 2t,2t+1   <- k = 16t+j, +4
        a1[j] = (r.wb.x >> (4 * j)) & kNibPair;  // row g+8, cols 2t,2t+1
        a2[j] = (r.wa.y >> (4 * j)) & kNibPair;  // row g,   cols 2t+8,2t+9 <- k = 16t+8+j, +4
        a3[j] = (r.wb.y >> (4 * j)) & kNibPair;  // row g+8, cols 2t+8,2t+9
    }
    const float sa = h2f(r.sa), sb = h2f(r.sb), ba = h2f(r.ba), bb = h2f(r.bb);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int c = nt * 8 + lg;
        uint4 f0 = make_uint4(0, 0, 0, 0), f1 = make_uint4(0, 0, 0, 0);
        if (c < M) {
            f0 = reinterpret_cast<const uint4 *>(xf)[((gl * 2 + 0) * M + c) * 4 + lt];
            f1 = reinterpret_cast<const uint4 *>(xf)[((gl * 2 + 1) * M + c) * 4 + lt];
        }
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        mma_16816(d, a0[0], a1[0], a2[0], a3[0], f0.x, f0.y);
        mma_16816(d, a0[1], a1[1], a2[1], a3[1], f0.z, f0.w);
        mma_16816(d, a0[2], a1[2], a2[2], a3[2], f1.x, f1.y);
        mma_16816(d, a0[3], a1[3], a2[3], a3[3], f1.z, f1.w);
        const int c0 = nt * 8 + 2 * lt;
        const float X0 = (c0 < M) ? xsum[gl * M + c0] : 0.f;
        const float X1 = (c0 + 1 < M) ? xsum[gl * M + c0 + 1] : 0.f;
        acc.s[nt][0] = fmaf(sa, d[0], acc.s[nt][0]);
        acc.s[nt][1] = fmaf(sa, d[1], acc.s[nt][1]);
        acc.s[nt][2] = fmaf(sb, d[2], acc.s[nt][2]);
        acc.s[nt][3] = fmaf(sb, d[3], acc.s[nt][3]);
        acc.b[nt][0] = fmaf(ba, X0, acc.b[nt][0]);
        acc.b[nt][1] = fmaf(ba, X1, acc.b[nt][1]);
        acc.b[nt][2] = fmaf(bb, X0, acc.b[nt][2]);
        acc.b[nt][3] = fmaf(bb, X1, acc.b[nt][3]);
    }
}

// Dot products of the warp's 16-row tile with the staged activations over
// groups [wg0, wg1) (global group indices; xf/xsum hold groups from g0 on).
// Two batches of kUnroll groups are kept in flight.
template <int NT>
__device__ __forceinline__ void tile_dot(Acc<NT> &acc, const RowPtrs &p, int wg0, int wg1, int g0,
                                         const uint32_t *xf, const float *xsum, int M, int lg, int lt,
                                         GroupRegs (&bufA)[kUnroll], bool preloaded) {
    GroupRegs bufB[kUnroll];
    if (wg0 >= wg1) return;
    if (!preloaded) {
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) load_group(bufA[u], p, min(wg0 + u, wg1 - 1));
    }
    for (int gb = wg0; gb < wg1; gb += 2 * kUnroll) {
        if (gb + kUnroll < wg1) {
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) load_group(bufB[u], p, min(gb + kUnroll + u, wg1 - 1));
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
            if (gb + u < wg1) group_step<NT>(acc, bufA[u], xf, xsum, gb + u - g0, M, lg, lt);
        if (gb + 2 * kUnroll < wg1) {
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) load_group(bufA[u], p, min(gb + 2 * kUnroll + u, wg1 - 1));
        }
        if (gb + kUnroll < wg1) {
#pragma unroll
            for (int u = 0; u < kUnroll; ++u)
                if (gb + kUnroll + u < wg1)
                    group_step<NT>(acc, bufB[u], xf, xsum, gb + kUnroll + u - g0, M, lg, lt);
        }
    }
}

__device__ __forceinline__ RowPtrs row_ptrs(const uint32_t *qw, const uint16_t *sc, const uint16_t *bi,
                                            int row0, int N, int K, int lg, int lt) {
    const int ng = K / kGroup;
    const int ra = min(row0 + lg, N - 1), rb = min(row0 + lg + 8, N - 1);
    RowPtrs p;
    p.qa = qw + (size_t)ra * (K / 8) + 2 * lt;
    p.qb = qw + (size_t)rb * (K / 8) + 2 * lt;
    p.sa = sc + (size_t)ra * ng;
    p.sb = sc + (size_t)rb * ng;
    p.ba = bi + (size_t)ra * ng;
    p.bb = bi + (size_t)rb * ng;
    return p;
}

// Final value of accumulator element i of activation tile nt.
template <int NT>
__device__ __forceinline__ float acc_value(const Acc<NT> &acc, int nt, int i) {
    return fmaf(kTwo24, acc.s[nt][i], acc.b[nt][i]);
}

// ---------------------------------------------------------------------------
// w4_gemv kernel.  grid = (row tiles, C); cluster (1, C, 1) splits K.
// ---------------------------------------------------------------------------
template <int NT, int NW>
__global__ void __launch_bounds__(NW * 32)
    gemv_kernel(const uint16_t *__restrict__ x, const uint32_t *__restrict__ qw,
                const uint16_t *__restrict__ sc, const uint16_t *__restrict__ bi,
                uint16_t *__restrict__ y, int M, int N, int K, int gpc) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int ng = K / kGroup;
    const int C = gridDim.y;
    const int cr = blockIdx.y;
    const int g0 = cr * gpc;
    const int g1 = min(ng, g0 + gpc);
    const int ngl = max(0, g1 - g0);
    const int row0 = blockIdx.x * kTileRows;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int lg = lane >> 2, lt = lane & 3;

    uint32_t *xf = reinterpret_cast<uint32_t *>(smem);
    float *xsum = reinterpret_cast<float *>(smem + (size_t)ngl * M * 128);
    float *red = xsum + ngl * M;               // [NW][16][M]
    float *cpart = red + NW * kTileRows * M;   // [16][M]

    const int wg0 = g0 + (ngl * warp) / NW;
    const int wg1 = g0 + (ngl * (warp + 1)) / NW;
    const RowPtrs p = row_ptrs(qw, sc, bi, row0, N, K, lg, lt);

    // Start the weight stream before the activations are staged.
    GroupRegs bufA[kUnroll];
    if (wg0 < wg1) {
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) load_group(bufA[u], p, min(wg0 + u, wg1 - 1));
    }
    stage_activations(x, M, K, g0, ngl, xf, xsum);
    __syncthreads();

    Acc<NT> acc;
    acc.zero();
    tile_dot<NT>(acc, p, wg0, wg1, g0, xf, xsum, M, lg, lt, bufA, true);

#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int row = lg + ((i & 2) ? 8 : 0);
            const int col = nt * 8 + 2 * lt + (i & 1);
            if (col < M) red[(warp * kTileRows + row) * M + col] = acc_value<NT>(acc, nt, i);
        }
    __syncthreads();

    const int nout = kTileRows * M;  // up to 256 outputs, more than the CTA's threads
    if (C == 1) {
        for (int e = threadIdx.x; e < nout; e += blockDim.x) {
            float part = 0.f;
            for (int w = 0; w < NW; ++w) part += red[w * nout + e];
            const int row = e / M, col = e % M;
            if (row0 + row < N) y[(size_t)col * N + row0 + row] = __half_as_ushort(__float2half_rn(part));
        }
        return;
    }
    for (int e = threadIdx.x; e < nout; e += blockDim.x) {
        float part = 0.f;
        for (int w = 0; w < NW; ++w) part += red[w * nout + e];
        cpart[e] = part;
    }
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    if (cr == 0) {
        for (int e = threadIdx.x; e < nout; e += blockDim.x) {
            float tot = 0.f;
            for (int r = 0; r < C; ++r) tot += cluster.map_shared_rank(cpart, r)[e];
            const int row = e / M, col = e % M;
            if (row0 + row < N) y[(size_t)col * N + row0 + row] = __half_as_ushort(__float2half_rn(tot));
        }
    }
    cluster.sync();
}

// ---------------------------------------------------------------------------
// Token selection keys: order by (value desc, index asc) as one uint64.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t make_key(float v, int idx) {
    const uint32_t u = __float_as_uint(v + 0.0f);  // -0 -> +0
    const uint32_t hi = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ((uint64_t)hi << 32) | (uint64_t)(0xFFFFFFFFu - (uint32_t)idx);
}

__device__ __forceinline__ void decode_key(uint64_t key, float &v, int &idx) {
    const uint32_t hi = (uint32_t)(key >> 32);
    const uint32_t u = (hi & 0x80000000u) ? (hi & 0x7FFFFFFFu) : ~hi;
    v = __uint_as_float(u);
    idx = (int)(0xFFFFFFFFu - (uint32_t)key);
}

__device__ __forceinline__ uint64_t shfl_max_u64(uint64_t v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const uint64_t w = __shfl_xor_sync(0xffffffffu, v, o);
        v = w > v ? w : v;
    }
    return v;
}

// Block-wide maximum of one key per thread (blockDim multiple of 32, <= 1024).
__device__ uint64_t block_max_u64(uint64_t v, uint64_t *scratch) {
    v = shfl_max_u64(v);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    const int nw = blockDim.x >> 5;
    v = (threadIdx.x < nw) ? scratch[threadIdx.x] : 0ull;
    if (warp == 0) v = shfl_max_u64(v);
    if (threadIdx.x == 0) scratch[0] = v;
    __syncthreads();
    v = scratch[0];
    __syncthreads();
    return v;
}

// In-place descending bitonic sort of P (power of two) keys in shared memory.
__device__ void bitonic_sort_desc(uint64_t *keys, int P) {
    for (int size = 2; size <= P; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = threadIdx.x; i < (P >> 1); i += blockDim.x) {
                const int lo = 2 * stride * (i / stride) + (i % stride);
                const int hi = lo + stride;
                const bool desc = (lo & size) == 0;
                const uint64_t a = keys[lo], b = keys[hi];
                if ((a < b) == desc) {
                    keys[lo] = b;
                    keys[hi] = a;
                }
            }
            __syncthreads();
        }
    }
}

__host__ __device__ inline int pow2_at_least(int v) {
    int p = 1;
    while (p < v) p <<= 1;
    return p;
}

__host__ __device__ inline size_t align16(size_t v) { return (v + 15) & ~(size_t)15; }

// Shared-memory layout of lm_head pass 1 (byte offsets, 16-byte aligned).
struct LmSmem {
    size_t xsum, logits, keys, total;
};

__host__ __device__ inline LmSmem lm_smem_layout(int ng, int M, int rpc, int k) {
    LmSmem l;
    l.xsum = align16((size_t)ng * M * 128);
    l.logits = align16(l.xsum + (size_t)ng * M * 4);
    l.keys = align16(l.logits + (size_t)M * rpc * 4);
    l.total = l.keys + (size_t)pow2_at_least(rpc > k ? rpc : k) * 8;
    return l;
}

// ---------------------------------------------------------------------------
// lm_head pass 1: CTA b computes the logits of rows [b*rpc, (b+1)*rpc) into
// shared memory and writes its k best keys per activation row to
// ws[(m*G + b)*k + i].
// ---------------------------------------------------------------------------
template <int NT, int NW>
__global__ void __launch_bounds__(NW * 32)
    lmhead_pass1(const uint16_t *__restrict__ x, const uint32_t *__restrict__ qw,
                 const uint16_t *__restrict__ sc, const uint16_t *__restrict__ bi, int M, int N,
                 int K, int k, int rpc, uint64_t *__restrict__ ws) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int ng = K / kGroup;
    const int G = gridDim.x;
    const int n0 = blockIdx.x * rpc;
    const int n1 = min(N, n0 + rpc);
    const int rows = max(0, n1 - n0);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int lg = lane >> 2, lt = lane & 3;
    const int P = pow2_at_least(max(rpc, k));

    const LmSmem lay = lm_smem_layout(ng, M, rpc, k);
    uint32_t *xf = reinterpret_cast<uint32_t *>(smem);
    float *xsum = reinterpret_cast<float *>(smem + lay.xsum);
    float *lgt = reinterpret_cast<float *>(smem + lay.logits);     // [M][rpc]
    uint64_t *keys = reinterpret_cast<uint64_t *>(smem + lay.keys);  // [P]

    const int ntiles = (rows + kTileRows - 1) / kTileRows;
    GroupRegs bufA[kUnroll];
    bool preloaded = false;
    if (warp < ntiles) {
        const RowPtrs p = row_ptrs(qw, sc, bi, n0 + warp * kTileRows, N, K, lg, lt);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) load_group(bufA[u], p, min(u, ng - 1));
        preloaded = true;
    }
    stage_activations(x, M, K, 0, ng, xf, xsum);
    __syncthreads();

    for (int tile = warp; tile < ntiles; tile += NW) {
        const int row0 = n0 + tile * kTileRows;
        const RowPtrs p = row_ptrs(qw, sc, bi, row0, N, K, lg, lt);
        Acc<NT> acc;
        acc.zero();
        tile_dot<NT>(acc, p, 0, ng, 0, xf, xsum, M, lg, lt, bufA, preloaded);
        preloaded = false;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int row = row0 + lg + ((i & 2) ? 8 : 0);
                const int col = nt * 8 + 2 * lt + (i & 1);
                if (col < M && row < n1) lgt[col * rpc + (row - n0)] = acc_value<NT>(acc, nt, i);
            }
    }
    __syncthreads();

    for (int m = 0; m < M; ++m) {
        uint64_t *out = ws + ((size_t)m * G + blockIdx.x) * k;
        if (k == 1) {
            uint64_t best = 0ull;
            for (int i = threadIdx.x; i < rows; i += blockDim.x) {
                const uint64_t key = make_key(lgt[m * rpc + i], n0 + i);
                best = key > best ? key : best;
            }
            best = block_max_u64(best, keys);
            if (threadIdx.x == 0) out[0] = best;
        } else {
            for (int i = threadIdx.x; i < P; i += blockDim.x)
                keys[i] = (i < rows) ? make_key(lgt[m * rpc + i], n0 + i) : 0ull;
            __syncthreads();
            bitonic_sort_desc(keys, P);
            for (int i = threadIdx.x; i < k; i += blockDim.x) out[i] = keys[i];
            __syncthreads();
        }
    }
}

// lm_head pass 2: one CTA per activation row merges the G*k candidates.
__global__ void __launch_bounds__(1024)
    lmhead_pass2(const uint64_t *__restrict__ ws, int G, int k, int32_t *__restrict__ idx,
                 float *__restrict__ val) {
    extern __shared__ __align__(16) uint8_t smem[];
    uint64_t *keys = reinterpret_cast<uint64_t *>(smem);
    const int m = blockIdx.x;
    const int n = G * k;
    const uint64_t *src = ws + (size_t)m * n;
    if (k == 1) {
        uint64_t best = 0ull;
        for (int i = threadIdx.x; i < n; i += blockDim.x) best = src[i] > best ? src[i] : best;
        best = block_max_u64(best, keys);
        if (threadIdx.x == 0) {
            float v;
            int id;
            decode_key(best, v, id);
            idx[m] = id;
            val[m] = v;
        }
        return;
    }
    const int P = pow2_at_least(n);
    for (int i = threadIdx.x; i < P; i += blockDim.x) keys[i] = (i < n) ? src[i] : 0ull;
    __syncthreads();
    bitonic_sort_desc(keys, P);
    for (int i = threadIdx.x; i < k; i += blockDim.x) {
        float v;
        int id;
        decode_key(keys[i], v, id);
        idx[(size_t)m * k + i] = id;
        val[(size_t)m * k + i] = v;
    }
}

// ---------------------------------------------------------------------------
// Host-side planning.
// ---------------------------------------------------------------------------
constexpr int kGemvWarps = 4;
constexpr int kLmWarps = 16;
constexpr int kMaxSmem = 227 * 1024;
constexpr int kMaxCandidates = 16384;  // pass-2 sort size (keys)

struct GemvPlan {
    int C;      // CTAs per cluster splitting K
    int gpc;    // groups per CTA
    size_t smem;
};

size_t gemv_smem(int ngl, int M) {
    return (size_t)ngl * M * 128 + (size_t)ngl * M * 4 + (size_t)kGemvWarps * kTileRows * M * 4 +
           (size_t)kTileRows * M * 4;
}

GemvPlan plan_gemv(int M, int N, int K) {
    const int ng = K / kGroup;
    const int rt = (N + kTileRows - 1) / kTileRows;
    const int target = 2 * sm_count();
    GemvPlan pl{1, ng, 0};
    int C = 1;
    while (C < 8 && rt * C < target && ng / (2 * C) >= kGemvWarps) C *= 2;
    // Keep the staged activations within shared memory.
    while (C < 8 && gemv_smem((ng + C - 1) / C, M) > (size_t)kMaxSmem / 2) C *= 2;
    pl.C = C;
    pl.gpc = (ng + C - 1) / C;
    pl.smem = gemv_smem(pl.gpc, M);
    return pl;
}

// Raise a kernel's dynamic shared-memory limit once per device (and only
// upwards), so that launches captured into CUDA graphs issue no attribute calls.
template <typename Kern>
bool ensure_smem(Kern kern, size_t bytes) {
    static size_t granted[64] = {0};
    if (bytes <= 48 * 1024) return true;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    if (granted[dev] >= bytes) return true;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) != cudaSuccess)
        return false;
    granted[dev] = bytes;
    return true;
}

template <int NT>
int launch_gemv(const uint16_t *x, const uint32_t *qw, const uint16_t *sc, const uint16_t *bi,
                uint16_t *y, int M, int N, int K, cudaStream_t st) {
    const GemvPlan pl = plan_gemv(M, N, K);
    if (pl.smem > (size_t)kMaxSmem) return W4_ERR_SHAPE;
    auto kern = gemv_kernel<NT, kGemvWarps>;
    if (!ensure_smem(kern, pl.smem)) return W4_ERR_LAUNCH;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((N + kTileRows - 1) / kTileRows, pl.C, 1);
    cfg.blockDim = dim3(kGemvWarps * 32, 1, 1);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = pl.C;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pl.C > 1 ? 1 : 0;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, x, qw, sc, bi, y, M, N, K, pl.gpc);
    return e == cudaSuccess ? W4A16_OK : W4_ERR_LAUNCH;
}

struct LmPlan {
    int G, rpc;
    size_t smem1, smem2;
};

bool plan_lmhead(int M, int N, int K, int k, int sms, LmPlan &pl) {
    const int ng = K / kGroup;
    const int max_rpc = 16384 / M;  // logits buffer <= 64 KB
    int rpc = (N + sms - 1) / sms;
    rpc = ((rpc + kTileRows - 1) / kTileRows) * kTileRows;
    const int min_rpc_cand = (int)(((long long)N * k + kMaxCandidates - 1) / kMaxCandidates);
    if (rpc < min_rpc_cand) rpc = ((min_rpc_cand + kTileRows - 1) / kTileRows) * kTileRows;
    if (rpc > max_rpc) return false;
    pl.rpc = rpc;
    pl.G = (N + rpc - 1) / rpc;
    if ((long long)pl.G * k > kMaxCandidates) return false;
    pl.smem1 = lm_smem_layout(ng, M, rpc, k).total;
    pl.smem2 = (size_t)(k == 1 ? 32 : pow2_at_least(pl.G * k)) * 8;
    return pl.smem1 <= (size_t)kMaxSmem && pl.smem2 <= (size_t)kMaxSmem;
}

// Upper bound on the pass-1 grid for a given (N, k), independent of the GPU.
long long lm_max_blocks(int N, int k) {
    const long long tiles = (N + kTileRows - 1) / kTileRows;
    const long long cap = kMaxCandidates / k;
    return tiles < cap ? tiles : cap;
}

template <int NT>
int launch_lmhead(const uint16_t *x, const uint32_t *qw, const uint16_t *sc, const uint16_t *bi, int M,
                  int N, int K, int k, int32_t *idx, float *val, uint64_t *ws, const LmPlan &pl,
                  cudaStream_t st) {
    auto k1 = lmhead_pass1<NT, kLmWarps>;
    if (!ensure_smem(k1, pl.smem1) || !ensure_smem(lmhead_pass2, pl.smem2)) return W4_ERR_LAUNCH;
    k1<<<pl.G, kLmWarps * 32, pl.smem1, st>>>(x, qw, sc, bi, M, N, K, k, pl.rpc, ws);
    if (cudaGetLastError() != cudaSuccess) return W4_ERR_LAUNCH;
    lmhead_pass2<<<M, 1024, pl.smem2, st>>>(ws, pl.G, k, idx, val);
    return launch_status();
}

int check_common(const void *x, const uint32_t *qw, const uint16_t *sc, const uint16_t *bi, int M, int N,
                 int K, int group) {
    if (!x || !qw || !sc || !bi) return W4_ERR_NULL;
    if (group != kGroup) return W4_ERR_GROUP;
    if (M < 1 || M > 16 || N < 1 || K < kGroup || K % kGroup != 0) return W4_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(qw) || !aligned16(sc) || !aligned16(bi)) return W4_ERR_ALIGN;
    return W4A16_OK;
}

}  // namespace
}  // namespace w4a16

using namespace w4a16;

extern "C" int w4_gemv(const uint16_t *x, const uint32_t *qweight, const uint16_t *scales,
                       const uint16_t *biases, uint16_t *y, int M, int N, int K, int group,
                       void *stream) {
    int st = check_common(x, qweight, scales, biases, M, N, K, group);
    if (st != W4A16_OK) return st;
    if (!y) return W4_ERR_NULL;
    if (!aligned16(y)) return W4_ERR_ALIGN;
    if (gemv_smem((K / kGroup + 7) / 8, M) > (size_t)kMaxSmem) return W4_ERR_SHAPE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return M <= 8 ? launch_gemv<1>(x, qweight, scales, biases, y, M, N, K, s)
                  : launch_gemv<2>(x, qweight, scales, biases, y, M, N, K, s);
}

extern "C" size_t lm_head_workspace_bytes(int M, int N, int k) {
    if (M < 1 || M > 16 || N < 1 || k < 1 || k > 64 || k > N) return 0;
    if ((long long)N * k > 16777216LL) return 0;
    return (size_t)M * (size_t)lm_max_blocks(N, k) * (size_t)k * sizeof(uint64_t);
}

extern "C" int lm_head_argmax_topk(const uint16_t *x, const uint32_t *qweight, const uint16_t *scales,
                                   const uint16_t *biases, int M, int N, int K, int group, int k,
                                   int32_t *idx, float *val, void *workspace, size_t workspace_bytes,
                                   void *stream) {
    int st = check_common(x, qweight, scales, biases, M, N, K, group);
    if (st != W4A16_OK) return st;
    if (!idx || !val) return W4_ERR_NULL;
    if (k < 1 || k > 64 || k > N || (long long)N * k > 16777216LL) return W4_ERR_SHAPE;
    if (!aligned16(idx) || !aligned16(val)) return W4_ERR_ALIGN;
    const size_t need = lm_head_workspace_bytes(M, N, k);
    if (!workspace || workspace_bytes < need) return W4_ERR_WORKSPACE;
    if (!aligned16(workspace)) return W4_ERR_ALIGN;
    LmPlan pl;
    if (!plan_lmhead(M, N, K, k, sm_count(), pl)) return W4_ERR_SHAPE;
    if ((long long)pl.G > lm_max_blocks(N, k)) return W4_ERR_SHAPE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint64_t *ws = reinterpret_cast<uint64_t *>(workspace);
    return M <= 8 ? launch_lmhead<1>(x, qweight, scales, biases, M, N, K, k, idx, val, ws, pl, s)
                  : launch_lmhead<2>(x, qweight, scales, biases, M, N, K, k, idx, val, ws, pl, s);
}

// ---------------------------------------------------------------------------
// lm_head_argmax_topk_noalloc: the same two kernels, with their candidate
// buffer in a fixed device array owned by this library instead of a caller
// workspace.  It exists for callers that cannot allocate device memory at the
// point of the call: code running inside a memory-pool or allocator callback,
// a host with a fixed memory budget, or an embedding that owns no allocator at
// all.  The array is static: every GPU that loads this library keeps it until
// the process exits.
// ---------------------------------------------------------------------------
namespace w4a16 {
namespace {

// 2 MiB: M <= 16 rows x at most 16384 candidate keys of 8 bytes, i.e. every
// size lm_head_argmax_topk accepts.
constexpr size_t kNoAllocScratchBytes = (size_t)16 * kMaxCandidates * sizeof(uint64_t);
static __device__ __align__(256) uint64_t g_lm_scratch[kNoAllocScratchBytes / sizeof(uint64_t)];

// Device address of g_lm_scratch for the current device.  The host-side name
// is only a stand-in; the address is looked up once per device and cached.
void *noalloc_scratch() {
    static std::mutex mu;
    static void *addr[64] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_lm_scratch) != cudaSuccess) return nullptr;
        addr[dev] = p;
    }
    return addr[dev];
}

}  // namespace
}  // namespace w4a16

extern "C" int lm_head_argmax_topk_noalloc(const uint16_t *x, const uint32_t *qweight,
                                           const uint16_t *scales, const uint16_t *biases, int M, int N,
                                           int K, int group, int k, int32_t *idx, float *val,
                                           void *stream) {
    int st = check_common(x, qweight, scales, biases, M, N, K, group);
    if (st != W4A16_OK) return st;
    if (!idx || !val) return W4_ERR_NULL;
    if (k < 1 || k > 64 || k > N || (long long)N * k > 16777216LL) return W4_ERR_SHAPE;
    if (!aligned16(idx) || !aligned16(val)) return W4_ERR_ALIGN;
    const size_t need = lm_head_workspace_bytes(M, N, k);
    if (need == 0 || need > kNoAllocScratchBytes) return W4_ERR_WORKSPACE;
    void *scratch = noalloc_scratch();
    if (!scratch) return W4_ERR_DEVICE;
    LmPlan pl;
    if (!plan_lmhead(M, N, K, k, sm_count(), pl)) return W4_ERR_SHAPE;
    if ((long long)pl.G > lm_max_blocks(N, k)) return W4_ERR_SHAPE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint64_t *ws = reinterpret_cast<uint64_t *>(scratch);
    return M <= 8 ? launch_lmhead<1>(x, qweight, scales, biases, M, N, K, k, idx, val, ws, pl, s)
                  : launch_lmhead<2>(x, qweight, scales, biases, M, N, K, k, idx, val, ws, pl, s);
}
