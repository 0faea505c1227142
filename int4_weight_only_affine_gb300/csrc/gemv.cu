// Decode-side kernels: the W4A16 multi-row GEMV (w4_gemv) and the LM-head
// GEMV fused with greedy / top-k token selection (lm_head_argmax_topk).
//
// "The inference engine - Mojo 1.0 on Metal", "Crossing Mojo 1.0": the decode
// GEMV is weight-streaming bound; each worker owns several output rows and
// keeps independent weight streams in flight, and token selection runs on the
// device so no logits vector is downloaded.
//
// Design (sm_103a): one streaming kernel serves both calls.
//  * Persistent CTAs (at most one per SM), each owning a contiguous range of
//    16-row tiles and a K-slice of them.  Warp 8 is the producer: one thread
//    streams each tile's K-chunk (up to 32 groups) into a ring of shared
//    memory stages with TMA (16 rows x 128 B boxes, 128-byte swizzle) and
//    the tile's scales and biases with one contiguous bulk copy each; stage
//    completion is counted on mbarriers (bounded waits).  Up to ~100 KB per
//    SM are in flight without holding registers.
//  * Warps 0-7 consume: lane (g, t) reads words 2t, 2t+1 of a group for rows
//    g and g+8 (conflict-free under the swizzle) and unpacks them straight
//    into the A operand of an m16n8k16 tensor-core MMA: (word >> 4j) &
//    0x000F000F places codes j and j+4 in a half pair as binary16 subnormals
//    q * 2^-24, which are exact.  B holds up to 8 (or 16) activation rows,
//    pre-arranged in shared memory in fragment order.  Products are exact and
//    accumulate in fp32.
//  * The affine step is folded per group: with P = sum_{k in g} q x and
//    X = sum_{k in g} x,  sum_k w x = scale * P + bias * X; acc_s += scale *
//    (P * 2^-24), acc_b += bias * X, y = 2^24 * acc_s + acc_b.
//  * The 8 consumer warps split each tile's K-chunk; their partial sums are
//    combined in fixed order after one named barrier per tile.  Matrices with
//    few tiles also split K across a thread-block cluster (2-8 CTAs), whose
//    partials are combined once at the end through distributed shared memory.
//    Results are deterministic.
//  * Programmatic dependent launch: every CTA releases the next kernel at
//    once; the producer never waits on the previous kernel (weights are
//    constants), the consumers wait before reading activations and writing
//    outputs.  Launched without the attribute this is ordinary stream order.
#include <cooperative_groups.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "gemv_tile.cuh"
#include "../../include/w4a16_testing.h"

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

// Reads and clears this translation unit's expired-wait record.
int gemv_wait_flag() {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_wait_expired, sizeof(int)) != cudaSuccess) return -1;
    if (v) {
        const int zero = 0;
        cudaMemcpyToSymbol(g_wait_expired, &zero, sizeof(int));
    }
    return v;
}

namespace {

// ---------------------------------------------------------------------------
// Token selection keys: (value desc, index asc) as one uint64 so that larger
// keys rank first.
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

// ---------------------------------------------------------------------------
// Warp-level top-64 of 64-bit keys.  A warp holds a list of 64 keys sorted
// descending, element i = 32*r + lane in register v[r].  A bitonic network
// (compare-exchange stages over shuffles) sorts a chunk of 64 keys, and two
// sorted lists merge into the 64 largest of their union: the elementwise
// maximum of one list and the other reversed is a bitonic sequence holding
// the 64 largest, which six more stages sort.  No block barrier is involved.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t umax64(uint64_t a, uint64_t b) { return a > b ? a : b; }
__device__ __forceinline__ uint64_t umin64(uint64_t a, uint64_t b) { return a < b ? a : b; }

// Two keys of a lane: list elements lane (a) and 32 + lane (b).
struct Key2 {
    uint64_t a, b;
};

// One compare-exchange stage: pairs (i, i ^ stride) ordered descending when
// (i & size) == 0, ascending otherwise (the lower index keeps the larger key
// in a descending block).
__device__ __forceinline__ Key2 bitonic_stage64(Key2 v, int size, int stride, int lane) {
    if (stride == 32) {  // only in the last block (size 64): descending
        return Key2{umax64(v.a, v.b), umin64(v.a, v.b)};
    }
    const uint64_t oa = __shfl_xor_sync(0xffffffffu, v.a, stride);
    const uint64_t ob = __shfl_xor_sync(0xffffffffu, v.b, stride);
    const bool lower = (lane & stride) == 0;
    const bool keep_a = lower == ((lane & size) == 0);         // element lane
    const bool keep_b = lower == (((32 + lane) & size) == 0);  // element 32 + lane
    return Key2{keep_a ? umax64(v.a, oa) : umin64(v.a, oa), keep_b ? umax64(v.b, ob) : umin64(v.b, ob)};
}

// The networks are unrolled (every stage's size and stride are constants) in
// out-of-line functions: one copy of the code serves every call site.
__device__ __noinline__ Key2 warp_sort64(Key2 v, int lane) {
#pragma unroll
    for (int size = 2; size <= 64; size <<= 1)
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) v = bitonic_stage64(v, size, stride, lane);
    return v;
}

// The 64 largest of run and c (both sorted descending), sorted descending.
__device__ __noinline__ Key2 warp_merge64(Key2 run, Key2 c, int lane) {
    const uint64_t ra = __shfl_sync(0xffffffffu, c.b, 31 - lane);  // c[63 - i] for i = lane
    const uint64_t rb = __shfl_sync(0xffffffffu, c.a, 31 - lane);  // c[63 - i] for i = 32 + lane
    Key2 v{umax64(run.a, ra), umax64(run.b, rb)};
#pragma unroll
    for (int stride = 32; stride > 0; stride >>= 1) v = bitonic_stage64(v, 64, stride, lane);
    return v;
}

// The 64 largest of run and an unsorted chunk c.
__device__ __forceinline__ Key2 warp_insert64(Key2 run, Key2 c, int lane) {
    return warp_merge64(run, warp_sort64(c, lane), lane);
}

// Combines the sorted lists of nw warps (lists[w][64] in shared memory) into
// lists[0] with a pairwise tree; called by every thread of the block.
__device__ void block_merge_lists(uint64_t (*lists)[64], int nw) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int span = 1; span < nw; span <<= 1) {
        __syncthreads();
        // A sorted list that starts with 0 is empty: nothing to merge.
        if ((warp % (2 * span)) == 0 && warp + span < nw && lists[warp + span][0] != 0ull) {
            const Key2 run = warp_merge64(Key2{lists[warp][lane], lists[warp][32 + lane]},
                                          Key2{lists[warp + span][lane], lists[warp + span][32 + lane]}, lane);
            lists[warp][lane] = run.a;
            lists[warp][32 + lane] = run.b;
        }
    }
    __syncthreads();
}

// ---------------------------------------------------------------------------
// The streaming kernel.
// ---------------------------------------------------------------------------

// Everything a launch needs besides the weight tensor map.  Byte offsets are
// relative to the 1024-aligned start of dynamic shared memory.
struct StreamArgs {
    const uint16_t *x, *sc, *bi;
    uint16_t *y;   // w4_gemv: output [M][N]
    uint64_t *ws;  // lm_head pass 1: candidate keys [M][gridDim.x][k]
    int M, N, K, k;
    int C;       // CTAs per cluster splitting K
    int tiles;   // ceil(N / 16)
    int stages;  // ring depth
    int ng;      // groups (64-k blocks) along K
    WFmt f;      // scale layout (quantisation group, symmetric codes)
    int units;   // 8-group units along K
    int nq_full; // whole 128-byte quads (4 groups) per row
    int cq;      // quads per 3-D copy
    int defer;   // 1: per-warp partials of all tiles kept, combined once at the end
    uint32_t stage_bytes, w_bytes;
    uint32_t off_xf, off_xsum, off_red, off_res, off_bar;
};

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory"); }

// FMT: the scale-layout class of the weight (kFmtG64, kFmtS128, kFmtAny,
// kFmtG32).
template <int NT, bool LMHEAD, bool M1, int FMT>
__global__ void __launch_bounds__(kThreads, NT == 1 ? 2 : 1)
    stream_kernel(const __grid_constant__ CUtensorMap tm3, const __grid_constant__ CUtensorMap tm2,
                  const StreamArgs a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = (uint32_t)__cvta_generic_to_shared(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *sb = smem_raw + (base - raw);
    pdl_launch_dependents();

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int M = a.M, N = a.N, ng = a.ng, S = a.stages, C = a.C;
    const int rank = blockIdx.x % C;
    const int ncl = gridDim.x / C, cl = blockIdx.x / C;
    const int t0 = (int)((long long)cl * a.tiles / ncl);
    const int t1 = (int)((long long)(cl + 1) * a.tiles / ncl);
    const int ntl = t1 - t0;
    const int gs0 = 8 * (rank * a.units / C);
    const int gs1 = min(ng, 8 * ((rank + 1) * a.units / C));
    const int ngl = max(0, gs1 - gs0);
    const int nch = (ngl + kChunkGroups - 1) / kChunkGroups;
    const int out16 = kTileRows * M;

    uint32_t *xf = reinterpret_cast<uint32_t *>(sb + a.off_xf);
    float *xsum = reinterpret_cast<float *>(sb + a.off_xsum);
    float *red = reinterpret_cast<float *>(sb + a.off_red);  // [2][8][16*M]
    float *res = reinterpret_cast<float *>(sb + a.off_res);  // [ntl][16*M]
    const uint32_t bar0 = base + a.off_bar;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sb + a.off_bar + 16 * S);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), kConsumerWarps);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(&tm3) : "memory");
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ---------------- producer: weights need no dependency wait ----------------
        if (lane == 0) {
            uint32_t issued_ph = 0, issued_any = 0;
            int it = 0;
            bool ok = true;
            for (int tl = 0; tl < ntl && ok; ++tl) {
                const int t = t0 + tl;
                const bool tail = (t + 1) * kTileRows > N;
                for (int ch = 0; ch < nch; ++ch, ++it) {
                    const int s = it % S;
                    const uint32_t ph = (it / S) & 1;
                    if (!mbar_wait(empty_bar(s), ph ^ 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const int cg0 = gs0 + ch * kChunkGroups;
                    const int len = min(kChunkGroups, gs1 - cg0);
                    const int q0 = cg0 / kBoxGroups;
                    const int nbox = (len + kBoxGroups - 1) / kBoxGroups;
                    // The tile's scale rows (and bias rows) are contiguous: [16][ngs].
                    const bool sym = FMT == kFmtS128 || (FMT != kFmtG64 && a.f.sym);
                    const int ngs = FMT == kFmtG64 ? ng : FMT == kFmtS128 ? ng >> 1 : a.f.ngs;
                    const uint32_t sbytes = tail ? 0u : 32u * ngs;
                    const uint32_t sball = sym ? sbytes : 2 * sbytes;
                    const uint32_t st = base + s * a.stage_bytes;
                    if (q0 + nbox <= a.nq_full) {
                        // One 3-D copy: cq quads x 16 rows x 128 B, the same swizzled
                        // image as cq separate 16 x 128 B boxes.
                        mbar_expect_tx(full_bar(s), a.cq * kBoxBytes + sball);
                        tma_load_3d(st, &tm3, 0, t * kTileRows, q0, full_bar(s));
                    } else {
                        // The chunk holding the ragged end of a row: one box per quad.
                        mbar_expect_tx(full_bar(s), nbox * kBoxBytes + sball);
                        for (int b = 0; b < nbox; ++b)
                            tma_load_2d(st + b * kBoxBytes, &tm2, (q0 + b) * 32, t * kTileRows, full_bar(s));
                    }
                    if (!tail) {
                        bulk_load(st + a.w_bytes, a.sc + (size_t)t * kTileRows * ngs, sbytes, full_bar(s));
                        if (!sym)
                            bulk_load(st + a.w_bytes + sbytes, a.bi + (size_t)t * kTileRows * ngs, sbytes,
                                      full_bar(s));
                    }
                    issued_ph = (issued_ph & ~(1u << s)) | (ph << s);
                    issued_any |= 1u << s;
                }
            }
            // Every copy issued here has landed before the CTA moves on.
            for (int s = 0; s < S; ++s)
                if (issued_any & (1u << s)) mbar_wait(full_bar(s), (issued_ph >> s) & 1);
        }
    } else {
        // ---------------- consumers ----------------
        const int lg = lane >> 2, lt = lane & 3;
        // Warp w takes box w of every stage: groups 4w .. 4w+3 of the chunk.
        int off[4];
        box_offsets(off, warp, lg, lt);
        const int xoff = lane_xoff(M, lg, lt), xd1 = lane_xd1(M, lg);
        const int goff = FMT == kFmtG32 ? g32_offset(warp, lg, lt) : 0;
        WFmt f = a.f;
        // The fixed classes' layouts follow from ng (fewer live registers).
        if (FMT == kFmtG64) f.ngs = ng;
        if (FMT == kFmtS128) f.ngs = ng >> 1;
        const bool sym = FMT == kFmtS128 || (FMT != kFmtG64 && f.sym);
        const bool vec = FMT == kFmtG64 ? (ng & 3) == 0 : FMT == kFmtS128 ? (ng & 3) == 0 : box_vec_ok(f);
        pdl_wait();
        stage_activations<M1 ? 2 : 4, FMT == kFmtG32>(a.x, M, a.K, gs0, ngl, xf, xsum, tid, kConsumers);
        consumer_sync();
        int s = 0;
        uint32_t ph = 0;
        for (int tl = 0; tl < ntl; ++tl) {
            const int t = t0 + tl;
            const int row0 = t * kTileRows;
            const bool tail = row0 + kTileRows > N;
            Acc<NT> acc;
            acc.zero();
            for (int ch = 0; ch < nch; ++ch) {
                const bool ok = mbar_wait(full_bar(s), ph, abort_flag);
                const uint8_t *st = sb + (size_t)s * a.stage_bytes;
                uint16_t *sp = reinterpret_cast<uint16_t *>(sb + (size_t)s * a.stage_bytes + a.w_bytes);
                if (tail) {
                    // The producer copies no scales for the ragged last tile (its rows
                    // end inside the arrays); fill them here, rows past N repeated.
                    const int ngs = f.ngs;
                    for (int i = tid; i < (sym ? 1 : 2) * kTileRows * ngs; i += kConsumers) {
                        const int arr = i / (kTileRows * ngs), r = (i / ngs) % kTileRows, gi = i % ngs;
                        const uint16_t *src = arr ? a.bi : a.sc;
                        sp[i] = src[(size_t)min(row0 + r, N - 1) * ngs + gi];
                    }
                    fence_proxy_async_smem();  // a later bulk copy reuses these bytes
                    consumer_sync();
                }
                if (ok) {
                    const int g = gs0 + ch * kChunkGroups + kBoxGroups * warp;
                    const int n = min(kBoxGroups, gs1 - g);
                    const int gl = g - gs0;
                    const uint4 *xl = reinterpret_cast<const uint4 *>(xf) + (size_t)gl * 2 * M * 4 + xoff;
                    const float *xs = xsum + gl * M * (FMT == kFmtG32 ? 2 : 1);
                    if (n == kBoxGroups && vec)
                        box_mma<NT, M1, true, FMT>(acc, st, off, sp, f, g, n, xl, xd1, xs, M, lg, lt, goff);
                    else if (n > 0)
                        box_mma<NT, M1, false, FMT>(acc, st, off, sp, f, g, n, xl, xd1, xs, M, lg, lt, goff);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(empty_bar(s));
                if (++s == S) {
                    s = 0;
                    ph ^= 1;
                }
            }
            if (a.defer) {
                // Keep this warp's partial; all tiles are combined once at the end.
                float *mine = red + ((size_t)tl * kConsumerWarps + warp) * out16;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int row = lg + ((i & 2) ? 8 : 0);
                        const int col = nt * 8 + 2 * lt + (i & 1);
                        if (col < M) mine[row * M + col] = acc.template value<FMT == kFmtS128 ? -8 : 1>(nt, i);
                    }
                continue;
            }
            // Per-tile reduction over the 8 consumer warps, fixed order.
            float *mine = red + ((tl & 1) * kConsumerWarps + warp) * out16;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int row = lg + ((i & 2) ? 8 : 0);
                    const int col = nt * 8 + 2 * lt + (i & 1);
                    if (col < M) mine[row * M + col] = acc.template value<FMT == kFmtS128 ? -8 : 1>(nt, i);
                }
            consumer_sync();
            if (warp == (tl & (kConsumerWarps - 1))) {
                const float *grp = red + (tl & 1) * kConsumerWarps * out16;
                for (int e = lane; e < out16; e += 32) {
                    float v = 0.f;
#pragma unroll
                    for (int w = 0; w < kConsumerWarps; ++w) v += grp[w * out16 + e];
                    if (!LMHEAD && C == 1) {
                        const int row = e / M, col = e % M;
                        if (row0 + row < N) a.y[(size_t)col * N + row0 + row] = __half_as_ushort(__float2half_rn(v));
                    } else {
                        res[tl * out16 + e] = v;
                    }
                }
            }
        }
        if (a.defer) {
            consumer_sync();
            for (int i = tid; i < ntl * out16; i += kConsumers) {
                const int tl = i / out16, e = i % out16;
                const float *grp = red + (size_t)tl * kConsumerWarps * out16;
                float v = 0.f;
#pragma unroll
                for (int w = 0; w < kConsumerWarps; ++w) v += grp[w * out16 + e];
                if (!LMHEAD && C == 1) {
                    const int row = e / M, col = e % M, r = (t0 + tl) * kTileRows + row;
                    if (r < N) a.y[(size_t)col * N + r] = __half_as_ushort(__float2half_rn(v));
                } else {
                    res[tl * out16 + e] = v;
                }
            }
        }
    }
    __syncthreads();

    if (!LMHEAD) {
        if (C > 1) {
            // Tile tl is finished by rank tl % C, summing the ranks in order.
            cg::cluster_group cluster = cg::this_cluster();
            cluster.sync();
            for (int tl = rank; tl < ntl; tl += C) {
                const int row0 = (t0 + tl) * kTileRows;
                for (int e = tid; e < out16; e += kThreads) {
                    float v = 0.f;
                    for (int q = 0; q < C; ++q) v += cluster.map_shared_rank(res, q)[tl * out16 + e];
                    const int row = e / M, col = e % M;
                    if (row0 + row < N) a.y[(size_t)col * N + row0 + row] = __half_as_ushort(__float2half_rn(v));
                }
            }
            cluster.sync();
        }
        return;
    }

    // ---------------- lm_head pass 1: k best keys of this CTA's rows ----------------
    // The keys of this CTA's rows, best first, padded with 0 (below every key).
    const int n0 = t0 * kTileRows;
    const int rows = min(N, t1 * kTileRows) - n0;
    uint64_t(*lists)[64] = reinterpret_cast<uint64_t(*)[64]>(sb);  // the ring is free now
    constexpr int kWarps = kThreads / 32;
    if (a.k == 1) {
        // Greedy selection: warp w takes activation rows w, w + 9, ...
        for (int m = warp; m < M; m += kWarps) {
            uint64_t best = 0ull;
            for (int i = lane; i < rows; i += 32) best = umax64(best, make_key(res[i * M + m], n0 + i));
            best = shfl_max_u64(best);
            if (lane == 0) a.ws[(size_t)m * gridDim.x + blockIdx.x] = best;
        }
        return;
    }
    for (int m = 0; m < M; ++m) {
        uint64_t *out = a.ws + ((size_t)m * gridDim.x + blockIdx.x) * a.k;
        {
            // Each warp keeps the best 64 of its 64-row chunks; a tree merges them.
            Key2 run{0ull, 0ull};
            for (int c0 = warp * 64; c0 < rows; c0 += kWarps * 64) {
                const int i = c0 + lane, j = c0 + 32 + lane;
                const Key2 c{i < rows ? make_key(res[i * M + m], n0 + i) : 0ull,
                             j < rows ? make_key(res[j * M + m], n0 + j) : 0ull};
                run = warp_insert64(run, c, lane);
            }
            lists[warp][lane] = run.a;
            lists[warp][32 + lane] = run.b;
            block_merge_lists(lists, kWarps);
            for (int i = tid; i < a.k; i += kThreads) out[i] = lists[0][i];
            __syncthreads();
        }
    }
}

// ---------------------------------------------------------------------------
// Projection-list kernel: a sequence of GEMVs in one persistent launch.
//
// "The inference engine - Mojo 1.0 on Metal", "Appendix: the remaining gap":
// the per-token floor of some 250 small launches is the binding constraint of
// decode.  Here one cooperative, persistent launch (one CTA per SM) runs a
// whole list of GEMVs.  The producer warp streams the weights of operation
// after operation into the ring without ever waiting for results (weights
// are constants), so HBM stays busy across operation boundaries; the 16
// consumer warps wait, where an operation's activations depend on earlier
// outputs, until every CTA has published the earlier operations (a counter
// in the caller's workspace, bounded spin), then stage the activations with
// coherent loads and compute as the streaming kernel does.  Each operation's
// tiles are split over the CTAs; outputs are combined in fixed order.
// ---------------------------------------------------------------------------
constexpr int kSeqMaxOps = 96;  // operations per launch (tensor maps travel as kernel parameters)
constexpr size_t kSeqCounterBytes = 16;  // workspace head: completion counter, epoch, finished CTAs
constexpr int kSeqWarps = 16;
constexpr int kSeqTeamWarps = 8;  // consumer warps per tile team
constexpr int kSeqConsumers = kSeqWarps * 32;
constexpr int kSeqThreads = kSeqConsumers + 32;

struct SeqOp {
    const uint16_t *x, *sc, *bi;
    uint16_t *y;
    const uint32_t *xt;  // tagged copy of x written earlier in this launch, or null
    uint32_t *yt;        // tagged copy of y for later operations, or null
    int N, K, wait_prev, cq;
    int src;             // operation (of this launch) that writes xt
    WFmt f;              // scale layout
};

struct SeqParams {
    CUtensorMap maps[kSeqMaxOps];  // 3-D code maps, one per operation
    SeqOp ops[kSeqMaxOps];
    unsigned *ws;                  // [0] (operation, CTA) completions, [1] launch epoch, [2] CTAs finished
    unsigned long long wait_ns;    // limit of a completion-counter wait
    unsigned target_bump;          // added to every counter target (0; nonzero only under the test hook)
    int nops, M, stages;
    int publish;                   // 1: some operation waits on the completion counter
    uint32_t stage_bytes, w_bytes;
    uint32_t off_xf, off_xsum, off_red, off_bar;
};

// 16-bit tag (1..65535) of the words operation `op` writes in the launch of
// epoch `epoch`: distinct for the operations of a launch and from those of the
// previous launch as long as nops < 65535.
__device__ __forceinline__ uint32_t seq_tag(unsigned epoch, int nops, int op) {
    return (uint32_t)(((unsigned long long)epoch * (unsigned)nops + (unsigned)op) % 65535ull) + 1u;
}

__device__ __forceinline__ void seq_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kSeqConsumers) : "memory"); }
// Named barrier of one 8-warp team (ids 2 and 3).
__device__ __forceinline__ void team_sync(int team) {
    asm volatile("bar.sync %0, %1;" ::"r"(2 + team), "n"(kSeqTeamWarps * 32) : "memory");
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// FMT: the scale-layout class shared by every operation of the launch (the
// host splits lists so).
template <int NT, bool M1, int FMT>
__global__ void __launch_bounds__(kSeqThreads, 1) seq_kernel(const __grid_constant__ SeqParams P) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = (uint32_t)__cvta_generic_to_shared(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *sb = smem_raw + (base - raw);
    pdl_launch_dependents();

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int M = P.M, S = P.stages, G = gridDim.x, blk = blockIdx.x;
    const int out16 = kTileRows * M;
    uint32_t *xf = reinterpret_cast<uint32_t *>(sb + P.off_xf);
    float *xsum = reinterpret_cast<float *>(sb + P.off_xsum);
    float *red = reinterpret_cast<float *>(sb + P.off_red);
    const uint32_t bar0 = base + P.off_bar;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sb + P.off_bar + 16 * S);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), kSeqTeamWarps);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    if (warp == kSeqWarps) {
        // ---------------- producer: streams every operation's weights ----------------
        if (lane == 0) {
            uint32_t issued_ph = 0, issued_any = 0;
            int it = 0;
            bool ok = true;
            for (int op = 0; op < P.nops && ok; ++op) {
                const SeqOp &o = P.ops[op];
                const int T = (o.N + kTileRows - 1) / kTileRows;
                const int t0 = (int)((long long)blk * T / G), t1 = (int)((long long)(blk + 1) * T / G);
                const int ng = o.K / kGroup, nch = (ng + kChunkGroups - 1) / kChunkGroups;
                for (int t = t0; t < t1 && ok; ++t) {
                    const bool tail = (t + 1) * kTileRows > o.N;
                    const bool sym = FMT == kFmtS128 || (FMT != kFmtG64 && o.f.sym);
                    const int ngs = FMT == kFmtG64 ? ng : FMT == kFmtS128 ? ng >> 1 : o.f.ngs;
                    const uint32_t sbytes = tail ? 0u : 32u * ngs;
                    const uint32_t sball = sym ? sbytes : 2 * sbytes;
                    for (int ch = 0; ch < nch; ++ch, ++it) {
                        const int s = it % S;
                        const uint32_t ph = (it / S) & 1;
                        if (!mbar_wait(empty_bar(s), ph ^ 1, abort_flag)) {
                            ok = false;
                            break;
                        }
                        const uint32_t st = base + s * P.stage_bytes;
                        mbar_expect_tx(full_bar(s), o.cq * kBoxBytes + sball);
                        tma_load_3d(st, &P.maps[op], 0, t * kTileRows, ch * (kChunkGroups / kBoxGroups), full_bar(s));
                        if (!tail) {
                            bulk_load(st + P.w_bytes, o.sc + (size_t)t * kTileRows * ngs, sbytes, full_bar(s));
                            if (!sym)
                                bulk_load(st + P.w_bytes + sbytes, o.bi + (size_t)t * kTileRows * ngs, sbytes,
                                          full_bar(s));
                        }
                        issued_ph = (issued_ph & ~(1u << s)) | (ph << s);
                        issued_any |= 1u << s;
                    }
                }
            }
            for (int s = 0; s < S; ++s)
                if (issued_any & (1u << s)) mbar_wait(full_bar(s), (issued_ph >> s) & 1);
        }
    } else {
        // ---------------- consumers: two teams of 8 warps, alternate tiles ----------------
        const int lg = lane >> 2, lt = lane & 3;
        const int team = warp / kSeqTeamWarps, tw = warp % kSeqTeamWarps;
        // Warp tw of a team takes box tw of every stage (groups 4tw .. 4tw+3).
        int off[4];
        box_offsets(off, tw, lg, lt);
        const int xoff = lane_xoff(M, lg, lt), xd1 = lane_xd1(M, lg);
        const int goff = FMT == kFmtG32 ? g32_offset(tw, lg, lt) : 0;
        // The workspace epoch counts completed launches; (epoch, operation)
        // names the 16-bit tag of every tagged word an operation writes, so a
        // word left by an earlier launch never matches.
        unsigned epoch;
        asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(epoch) : "l"(P.ws + 1) : "memory");
        pdl_wait();
        int base_it = 0;  // stages consumed by all earlier operations
        for (int op = 0; op < P.nops; ++op) {
            const SeqOp &o = P.ops[op];
            const int N = o.N, ng = o.K / kGroup, nch = (ng + kChunkGroups - 1) / kChunkGroups;
            // K % 256 == 0: every full box reads its scales as one vector.
            WFmt f = o.f;
            // The fixed classes' layouts follow from ng (fewer live registers).
            if (FMT == kFmtG64) f.ngs = ng;
            if (FMT == kFmtS128) f.ngs = ng >> 1;
            const bool sym = FMT == kFmtS128 || (FMT != kFmtG64 && f.sym);
            const int T = (N + kTileRows - 1) / kTileRows;
            const int t0 = (int)((long long)blk * T / G), t1 = (int)((long long)(blk + 1) * T / G);
            const int ntl = t1 - t0;
            if (o.wait_prev && op > 0 && !o.xt && tid == 0) {
                // Every CTA has published operations 0..op-1.
                const unsigned target = (unsigned)op * (unsigned)G + P.target_bump;
                const uint64_t t_start = global_ns();
                while (ld_acquire_u32(P.ws) < target) {
                    if (*abort_flag) break;
                    if (global_ns() - t_start > P.wait_ns) {
                        atomicExch(&g_wait_expired, 1);
                        *abort_flag = 1;
                        break;
                    }
                }
            }
            seq_sync();  // also ends every use of the previous operation's activations
            if (o.xt) {
                // Activations produced by an earlier operation of this launch: poll
                // the tagged words themselves (one L2 round trip, no counter).
                stage_activations_t<true, 2, FMT == kFmtG32>(nullptr, o.xt, seq_tag(epoch, P.nops, o.src), M, o.K, 0,
                                                             ng, xf, xsum, tid, kSeqConsumers, true, abort_flag);
            } else {
                stage_activations<2, FMT == kFmtG32>(o.x, M, o.K, 0, ng, xf, xsum, tid, kSeqConsumers, true);
            }
            seq_sync();
            // Tile tl, chunks ch0, ch0 + chs, ...; its 8 warps' partials go to
            // partial block `slot` (blocks of 8 warps x 16 x M).
            auto run_tile = [&](int tl, int ch0, int chs, int slot) {
                const int row0 = (t0 + tl) * kTileRows;
                const bool tail = row0 + kTileRows > N;
                Acc<NT> acc;
                acc.zero();
                // Stage index of this tile's first chunk: every earlier operation's
                // stages, then nch per earlier tile of this operation.
                const int it0 = base_it + tl * nch + ch0;
                int s = it0 % S;
                uint32_t ph = (it0 / S) & 1;
                for (int ch = ch0; ch < nch; ch += chs) {
                    const bool ok = mbar_wait(full_bar(s), ph, abort_flag);
                    const uint8_t *st = sb + (size_t)s * P.stage_bytes;
                    uint16_t *sp = reinterpret_cast<uint16_t *>(sb + (size_t)s * P.stage_bytes + P.w_bytes);
                    if (tail) {
                        // Only the last tile of the operation is ragged; its team
                        // fills the scales the producer could not copy.
                        const int ngs = f.ngs;
                        for (int i = tw * 32 + lane; i < (sym ? 1 : 2) * kTileRows * ngs; i += kSeqTeamWarps * 32) {
                            const int arr = i / (kTileRows * ngs), r = (i / ngs) % kTileRows, gi = i % ngs;
                            const uint16_t *src = arr ? o.bi : o.sc;
                            sp[i] = src[(size_t)min(row0 + r, N - 1) * ngs + gi];
                        }
                        fence_proxy_async_smem();  // a later bulk copy reuses these bytes
                        team_sync(team);
                    }
                    if (ok) {
                        const int g = ch * kChunkGroups + kBoxGroups * tw;
                        const int n = min(kBoxGroups, ng - g);
                        const uint4 *xl = reinterpret_cast<const uint4 *>(xf) + (size_t)g * 2 * M * 4 + xoff;
                        // (The sums' address is formed inside each call: this keeps the
                        // group-64 M = 1 variant within its 96 registers.)
                        constexpr int xsg = FMT == kFmtG32 ? 2 : 1;  // sums per group and row
                        if (n == kBoxGroups)
                            box_mma<NT, M1, true, FMT>(acc, st, off, sp, f, g, n, xl, xd1, xsum + g * M * xsg, M, lg,
                                                       lt, goff);
                        else if (n > 0)
                            box_mma<NT, M1, false, FMT>(acc, st, off, sp, f, g, n, xl, xd1, xsum + g * M * xsg, M, lg,
                                                        lt, goff);
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(empty_bar(s));
                    s += chs;  // chs <= 2 <= S: at most one wrap
                    if (s >= S) {
                        s -= S;
                        ph ^= 1;
                    }
                }
                float *mine = red + ((size_t)slot * kSeqTeamWarps + tw) * out16;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int row = lg + ((i & 2) ? 8 : 0);
                        const int col = nt * 8 + 2 * lt + (i & 1);
                        if (col < M) mine[row * M + col] = acc.template value<FMT == kFmtS128 ? -8 : 1>(nt, i);
                    }
            };
            // A CTA with a single tile of several chunks splits it by K (team
            // t takes chunks t, t + 2, ...: both teams work, partial blocks 0
            // and 1); otherwise the teams take alternate tiles.  Group-64
            // affine codes only: measured 1.2 % faster for a 3B decode list
            // in that class, 5 % slower in the symmetric group-128 class.
            constexpr bool kKSplit = FMT == kFmtG64;
            if (kKSplit && ntl == 1 && nch >= 2)
                run_tile(0, team, 2, team);
            else
                for (int tl = team; tl < ntl; tl += 2) run_tile(tl, 0, 1, tl);
            base_it += ntl * nch;
            seq_sync();
            for (int i = tid; i < ntl * out16; i += kSeqConsumers) {
                const int tl = i / out16, e = i % out16;
                const float *grp = red + (size_t)tl * kSeqTeamWarps * out16;
                float v = 0.f;
#pragma unroll
                for (int w = 0; w < kSeqTeamWarps; ++w) v += grp[w * out16 + e];
                if (kKSplit && ntl == 1 && nch >= 2)  // the other team's 8 partials of the single tile
#pragma unroll
                    for (int w = kSeqTeamWarps; w < 2 * kSeqTeamWarps; ++w) v += grp[w * out16 + e];
                const int row = e / M, col = e % M, r = (t0 + tl) * kTileRows + row;
                if (r < N) {
                    const uint16_t h = __half_as_ushort(__float2half_rn(v));
                    o.y[(size_t)col * N + r] = h;
                    if (o.yt) {
                        const uint32_t w = (seq_tag(epoch, P.nops, op) << 16) | h;
                        asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(o.yt + (size_t)col * N + r), "r"(w)
                                     : "memory");
                    }
                }
            }
            // Publish: the CTA barrier orders every thread's stores before the
            // signalling thread's release increment (cumulative at gpu scope).
            if (P.publish) {
                seq_sync();
                if (tid == 0) asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(P.ws) : "memory");
            }
        }
        if (tid == 0) {
            // The last CTA to finish resets the counters and advances the epoch
            // for the next launch on this workspace.
            __threadfence();
            if (atomicAdd(P.ws + 2, 1u) == (unsigned)G - 1u) {
                __threadfence();
                P.ws[0] = 0u;
                P.ws[2] = 0u;
                P.ws[1] = epoch + 1u;
            }
        }
    }
    __syncthreads();
}

template <int FMT>
const void *stream_kernel_ptr_f(int M, bool lmhead) {
    if (lmhead)
        return M == 1 ? (const void *)stream_kernel<1, true, true, FMT>
               : M <= 8 ? (const void *)stream_kernel<1, true, false, FMT>
                        : (const void *)stream_kernel<2, true, false, FMT>;
    return M == 1 ? (const void *)stream_kernel<1, false, true, FMT>
           : M <= 8 ? (const void *)stream_kernel<1, false, false, FMT>
                    : (const void *)stream_kernel<2, false, false, FMT>;
}

const void *stream_kernel_ptr(int M, bool lmhead, int fmt) {
    return fmt == kFmtG64    ? stream_kernel_ptr_f<kFmtG64>(M, lmhead)
           : fmt == kFmtS128 ? stream_kernel_ptr_f<kFmtS128>(M, lmhead)
           : fmt == kFmtG32  ? stream_kernel_ptr_f<kFmtG32>(M, lmhead)
                             : stream_kernel_ptr_f<kFmtAny>(M, lmhead);
}

// lm_head pass 2: one CTA per activation row merges the G*k candidates
// (G sorted lists of k keys).  Two lower bounds of the overall k-th key:
// the largest of the lists' k-th keys (its own list holds k keys above it)
// and the k-th largest of a subset of the lists' first keys (the best two
// that each lane of one warp sees; k lists each hold one key above it).  Only keys >= the larger bound T can be selected; for logits
// spread like independent samples about k of them remain.  They are
// compacted into shared memory (an overflow goes straight into the warps'
// running lists, so any input is handled), every warp keeps the best 64 of
// its chunks, and a tree merges the warps' lists.  Launched as a programmatic
// dependent of pass 1; it waits for pass 1's results first.
// Keys are distinct (the index is part of the key), so the rank of a key
// among a set is the number of larger keys: small sets (the lists' first
// keys, the survivors) are ranked by counting in shared memory.
// Number of keys in s[0..n) larger than key (shared memory, 8 loads in flight).
__device__ __forceinline__ int rank_of(uint64_t key, const uint64_t *s, int n) {
    int r = 0, j = 0;
    for (; j + 8 <= n; j += 8) {
        int c = 0;
#pragma unroll
        for (int u = 0; u < 8; ++u) c += s[j + u] > key;
        r += c;
    }
    for (; j < n; ++j) r += s[j] > key;
    return r;
}

constexpr int kPass2Threads = 1024;
constexpr int kSurvivorCap = 2048;
constexpr int kMaxPerThread = kMaxCandidates / kPass2Threads;  // candidates per row <= 16384
static_assert(kSurvivorCap >= kPass2Threads, "the survivor buffer first holds one first key per thread");

__global__ void __launch_bounds__(kPass2Threads)
    lmhead_pass2(const uint64_t *__restrict__ ws, int G, int k, int32_t *__restrict__ idx,
                 float *__restrict__ val) {
    __shared__ uint64_t lists[kPass2Threads / 32][64];
    __shared__ uint64_t buf[kSurvivorCap];
    __shared__ uint64_t scratch[kPass2Threads / 32];
    __shared__ unsigned nbuf;
    __shared__ unsigned fk_rank[kPass2Threads];
    pdl_wait();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    constexpr int kWarps = kPass2Threads / 32;
    const int m = blockIdx.x;
    const int n = G * k;
    const uint64_t *src = ws + (size_t)m * n;
    if (k == 1) {
        uint64_t best = 0ull;
        for (int i = tid; i < n; i += kPass2Threads) best = umax64(best, src[i]);
        best = block_max_u64(best, scratch);
        if (tid == 0) {
            float v;
            int id;
            decode_key(best, v, id);
            idx[m] = id;
            val[m] = v;
        }
        return;
    }
    // Every load is issued before any result is used: the candidates (at
    // most 16 per thread), the first key of list tid, and the k-th keys.
    uint64_t v[kMaxPerThread];
#pragma unroll
    for (int j = 0; j < kMaxPerThread; ++j) {
        const int i = tid + j * kPass2Threads;
        v[j] = i < n ? src[i] : 0ull;
    }
    const uint64_t fk = tid < G ? src[(size_t)tid * k] : 0ull;  // first key of list tid
    uint64_t t = 0ull;
    for (int c = tid; c < G; c += kPass2Threads) t = umax64(t, src[(size_t)c * k + k - 1]);
    uint64_t T = block_max_u64(t, scratch);
    if (G >= k) {
        // The k-th largest first key: k lists each hold a key at least that
        // large.  Keys are distinct, so counting the larger ones gives every
        // key its exact rank.
        buf[tid] = fk;
        fk_rank[tid] = 0u;
        if (tid == 0) scratch[0] = 0ull;
        __syncthreads();
        if (G <= kPass2Threads) {
            // P = 1024 / G threads count the larger first keys of list c,
            // each over a 1 / P share of the lists.
            const int P = kPass2Threads / G;
            if (tid < P * G) {
                const int c = tid % G, p = tid / G;
                const int j0 = p * G / P, j1 = (p + 1) * G / P;
                const uint64_t key = buf[c];
                int r = 0;
                for (int j = j0; j < j1; ++j) r += buf[j] > key;
                atomicAdd(&fk_rank[c], (unsigned)r);
            }
            __syncthreads();
            if (tid < G && fk_rank[tid] == (unsigned)(k - 1)) scratch[0] = fk;
        } else if (warp == 0) {
            // Many lists: a looser bound, the k-th largest of the best two
            // first keys each lane sees.
            uint64_t f0 = 0ull, f1 = 0ull;
            for (int c = lane; c < G; c += 32) {
                const uint64_t f = c < kPass2Threads ? buf[c] : src[(size_t)c * k];
                f1 = umax64(f1, umin64(f0, f));
                f0 = umax64(f0, f);
            }
            const Key2 best = warp_sort64(Key2{f0, f1}, lane);
            const uint64_t kth = __shfl_sync(0xffffffffu, (k - 1) < 32 ? best.a : best.b, (k - 1) & 31);
            if (lane == 0) scratch[0] = kth;
        }
        __syncthreads();
        T = umax64(T, scratch[0]);
        __syncthreads();
    }
    if (tid == 0) nbuf = 0u;
    __syncthreads();
    // Compact the keys >= T (one reservation per warp and register).
    Key2 run{0ull, 0ull};
#pragma unroll
    for (int j = 0; j < kMaxPerThread; ++j) {
        const uint64_t key = v[j] >= T ? v[j] : 0ull;
        const unsigned bal = __ballot_sync(0xffffffffu, key != 0ull);
        if (bal == 0u) continue;
        unsigned slot = 0;
        if (lane == 0) slot = atomicAdd(&nbuf, (unsigned)__popc(bal));
        slot = __shfl_sync(0xffffffffu, slot, 0);
        if (slot + __popc(bal) <= (unsigned)kSurvivorCap) {
            if (key) buf[slot + __popc(bal & ((1u << lane) - 1u))] = key;
        } else {
            // No room: keep them in this warp's list, and zero the reserved
            // slots that fall inside the buffer.
            if (slot + lane < (unsigned)kSurvivorCap && lane < __popc(bal)) buf[slot + lane] = 0ull;
            run = warp_insert64(run, Key2{key, 0ull}, lane);
        }
    }
    __syncthreads();
    if (nbuf <= (unsigned)kSurvivorCap) {
        // Every survivor is in buf: rank by counting, write the best k.
        const int nb = (int)nbuf;
        for (int i = tid; i < nb; i += kPass2Threads) {
            const uint64_t key = buf[i];
            const int r = rank_of(key, buf, nb);
            if (r < k) {
                float v;
                int id;
                decode_key(key, v, id);
                idx[(size_t)m * k + r] = id;
                val[(size_t)m * k + r] = v;
            }
        }
        return;
    }
    for (int c0 = warp * 64; c0 < kSurvivorCap; c0 += kWarps * 64)
        run = warp_insert64(run, Key2{buf[c0 + lane], buf[c0 + 32 + lane]}, lane);
    lists[warp][lane] = run.a;
    lists[warp][32 + lane] = run.b;
    block_merge_lists(lists, kWarps);
    for (int i = tid; i < k; i += kPass2Threads) {
        float v;
        int id;
        decode_key(lists[0][i], v, id);
        idx[(size_t)m * k + i] = id;
        val[(size_t)m * k + i] = v;
    }
}

// ---------------------------------------------------------------------------
// Host-side planning and launch.
// ---------------------------------------------------------------------------


// Upper bound on the pass-1 grid for a given (N, k), independent of the GPU.
long long lm_max_blocks(int N, int k) {
    const long long tiles = (N + kTileRows - 1) / kTileRows;
    const long long cap = kMaxCandidates / k;
    return tiles < cap ? tiles : cap;
}

struct StreamPlan {
    StreamArgs a;
    int grid;
    size_t smem;
};

// force_defer: keep every warp's partial of every tile (no per-tile barrier)
// even when that takes more than 32 KB.
bool layout_stream(StreamPlan &p, int M, bool lmhead, size_t ring_budget, int tpc, int slice_groups,
                   bool force_defer = false) {
    StreamArgs &a = p.a;
    const int wbox = min(kChunkGroups, slice_groups + kBoxGroups - 1) / kBoxGroups;
    const int xsums = a.f.gs == 0 ? 2 : 1;  // activation sums per group and row
    a.w_bytes = (uint32_t)(wbox * kBoxBytes);
    a.cq = wbox;
    a.nq_full = a.K / 256;
    // Codes, then the tile's scale rows [16][ngs] (and bias rows).
    a.stage_bytes = (uint32_t)align_up((size_t)a.w_bytes + (a.f.sym ? 32u : 64u) * a.f.ngs, 1024);
    // As many stages as the byte budget allows: the ring is what keeps HBM busy.
    const int stages = (int)max((size_t)2, min((size_t)kMaxStages, ring_budget / a.stage_bytes));
    a.stages = stages;
    size_t off = (size_t)stages * a.stage_bytes;
    if (lmhead) {
        // After the main loop the ring holds the selection keys.
        const size_t need = (size_t)(kThreads / 32) * 64 * 8;  // per-warp lists of the selection
        if (off < need) off = align_up(need, 1024);
    }
    a.off_xf = (uint32_t)off;
    off = align_up(off + (size_t)slice_groups * M * 128, 16);
    a.off_xsum = (uint32_t)off;
    off = align_up(off + (size_t)slice_groups * M * 4 * xsums, 16);
    a.off_red = (uint32_t)off;
    const size_t red_all = (size_t)tpc * kConsumerWarps * kTileRows * M * 4;
    a.defer = (force_defer || red_all <= 32 * 1024) ? 1 : 0;
    off = align_up(off + (a.defer ? red_all : (size_t)2 * kConsumerWarps * kTileRows * M * 4), 16);
    a.off_res = (uint32_t)off;
    if (lmhead || a.C > 1) off = align_up(off + (size_t)tpc * kTileRows * M * 4, 16);
    a.off_bar = (uint32_t)off;
    off += 16 * stages + 16;
    p.smem = off + 1024;  // alignment slack
    return true;
}

// CTAs per SM: two for up to 8 activation rows (16 consumer warps per SM and
// two rings in flight), one otherwise.
int ctas_per_sm(int M) { return M <= 8 ? 2 : 1; }

const void *stream_kernel_ptr(int M, bool lmhead, int fmt);
bool ensure_smem(const void *kern, size_t bytes);

// Clusters of C CTAs (this kernel, this shared memory) that can be resident
// at once; cached per (kernel, C, bytes, device).
int max_active_clusters(const void *kern, int C, size_t smem, int fallback) {
    struct Entry {
        const void *kern;
        int C, dev;
        size_t smem;
        int n;
    };
    static std::mutex mu;
    static Entry cache[128];
    static int n = 0;
    if (C == 1) return fallback;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return fallback;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n; ++i)
        if (cache[i].kern == kern && cache[i].C == C && cache[i].smem == smem && cache[i].dev == dev)
            return cache[i].n;
    int v = 0;
    if (!ensure_smem(kern, smem)) return fallback;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(C * 64, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&v, kern, &cfg) != cudaSuccess || v <= 0) {
        cudaGetLastError();
        v = fallback;
    }
    if (n < 128) cache[n++] = Entry{kern, C, dev, smem, v};
    return v;
}

// Lays out a launch with C CTAs per cluster; false if it does not fit.
// The largest layout within the per-CTA share of shared memory (false if
// none fits).
bool fit_layout(StreamPlan &p, bool lmhead, int per_sm, int tpc, int slice) {
    const size_t per_cta = (size_t)kMaxSmem / per_sm;
    // First choice: partials of all tiles kept (no per-tile barrier) with a
    // ring of at least 4 stages; else the largest layout that fits.
    for (size_t budget = per_cta; budget >= 16 * 1024; budget -= 8 * 1024) {
        layout_stream(p, p.a.M, lmhead, budget - (per_sm == 2 ? 24 * 1024 : 0), tpc, slice, true);
        if (p.smem <= per_cta) {
            if (p.a.stages >= 4) return true;
            break;
        }
    }
    for (size_t budget = per_cta; budget >= 16 * 1024; budget -= 8 * 1024) {
        layout_stream(p, p.a.M, lmhead, budget - (per_sm == 2 ? 24 * 1024 : 0), tpc, slice);
        if (p.smem <= per_cta) return true;
    }
    return false;
}

bool plan_with_cluster(StreamPlan &p, int C, int slots, int per_sm, bool lmhead) {
    StreamArgs &a = p.a;
    a.C = C;
    int ncl = min(a.tiles, max(1, slots / C));
    const int slice = min(a.ng, 8 * ((a.units + C - 1) / C));
    if (!fit_layout(p, lmhead, per_sm, (a.tiles + ncl - 1) / ncl, slice)) return false;
    if (C > 1) {
        // Keep every cluster resident: cap the cluster count by the occupancy
        // of the layout actually launched (fewer clusters mean more tiles per
        // cluster and possibly a larger layout, so check again).
        for (int iter = 0; iter < 3; ++iter) {
            const int act = max_active_clusters(stream_kernel_ptr(a.M, lmhead, fmt_class(a.f)), C, p.smem, ncl);
            if (act >= ncl) break;
            ncl = max(1, act);
            if (!fit_layout(p, lmhead, per_sm, (a.tiles + ncl - 1) / ncl, slice)) return false;
        }
    }
    p.grid = ncl * C;
    return true;
}

bool plan_stream(StreamPlan &p, int M, int N, int K, const WFmt &f, bool lmhead, int k) {
    StreamArgs &a = p.a;
    a.M = M;
    a.N = N;
    a.K = K;
    a.k = k;
    a.f = f;
    a.ng = K / kGroup;
    a.units = (a.ng + 7) / 8;
    a.tiles = (N + kTileRows - 1) / kTileRows;
    const int per_sm = ctas_per_sm(M);
    int slots = sm_count() * per_sm;
    if (lmhead) slots = min(slots, kMaxCandidates / k);
    // Split K over a cluster only when the tiles alone cannot spread evenly
    // over the SMs or the activations of a whole row do not fit (cost = work
    // of the busiest cluster in 16-row x 8-group units; a split must save at
    // least 10 %).
    int bestC = 0;
    long long bestCost = -1;
    for (int C = 1; C <= (lmhead ? 1 : 8); C *= 2) {
        if (C > a.units) break;
        StreamPlan trial = p;
        if (!plan_with_cluster(trial, C, slots, per_sm, lmhead)) continue;
        const int ncl = trial.grid / C;
        const long long cost = (long long)((a.tiles + ncl - 1) / ncl) * ((a.units + C - 1) / C);
        if (bestCost < 0 || cost * 10 < bestCost * 9) {
            bestC = C;
            bestCost = cost;
        }
    }
    if (bestC == 0) return false;
    return plan_with_cluster(p, bestC, slots, per_sm, lmhead);
}

// Raise a kernel's dynamic shared-memory limit once per (kernel, device), and
// only upwards, so that launches captured into CUDA graphs issue no attribute
// calls.
bool ensure_smem(const void *kern, size_t bytes) {
    struct Grant {
        const void *kern;
        int dev;
        size_t bytes;
    };
    static std::mutex mu;
    static Grant grants[64];
    static int ngrants = 0;
    if (bytes <= 48 * 1024) return true;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    std::lock_guard<std::mutex> lock(mu);
    int slot = -1;
    for (int i = 0; i < ngrants; ++i)
        if (grants[i].kern == kern && grants[i].dev == dev) slot = i;
    if (slot >= 0 && grants[slot].bytes >= bytes) return true;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) != cudaSuccess) {
        cudaGetLastError();  // leave no stale error for a later launch check
        return false;
    }
    if (slot < 0 && ngrants < 64) slot = ngrants++;
    if (slot >= 0) grants[slot] = Grant{kern, dev, bytes};
    return true;
}

template <int NT, bool LM, bool M1, int FMT>
int launch_stream(const StreamPlan &p, const uint32_t *qw, bool overlap, cudaStream_t st) {
    CUtensorMap tm3, tm2;
    const uint64_t KW = (uint64_t)p.a.K / 8;
    if (!make_map_2d(&tm2, CU_TENSOR_MAP_DATA_TYPE_UINT32, qw, KW, (uint64_t)p.a.N, KW * 4, 32, kTileRows,
                     CU_TENSOR_MAP_SWIZZLE_128B))
        return W4_ERR_DEVICE;
    if (p.a.nq_full > 0) {
        if (!make_map_3d(&tm3, CU_TENSOR_MAP_DATA_TYPE_UINT32, qw, 32, (uint64_t)p.a.N, (uint64_t)p.a.nq_full, KW * 4,
                         128, 32, kTileRows, (uint32_t)p.a.cq, CU_TENSOR_MAP_SWIZZLE_128B))
            return W4_ERR_DEVICE;
    } else {
        tm3 = tm2;  // never used: every chunk takes the 2-D path
    }
    auto kern = stream_kernel<NT, LM, M1, FMT>;
    if (!ensure_smem(reinterpret_cast<const void *>(kern), p.smem)) return W4_ERR_LAUNCH;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.grid, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (p.a.C > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = p.a.C;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    if (overlap) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, tm3, tm2, p.a);
    return e == cudaSuccess ? W4A16_OK : W4_ERR_LAUNCH;
}

// bi == nullptr: symmetric codes.  Fills the scale layout f.
int check_common(const void *x, const uint32_t *qw, const uint16_t *sc, const uint16_t *bi, int M, int N, int K,
                 int group, WFmt &f) {
    if (!x || !qw || !sc) return W4_ERR_NULL;
    if (M < 1 || M > 16 || N < 1 || K < kGroup || K % kGroup != 0) return W4_ERR_SHAPE;
    if (!make_fmt(f, K, group, bi == nullptr)) return W4_ERR_GROUP;
    if (!aligned16(x) || !aligned16(qw) || !aligned16(sc) || (bi && !aligned16(bi))) return W4_ERR_ALIGN;
    return W4A16_OK;
}

template <bool LM, int FMT>
int launch_stream_f(const StreamPlan &p, const uint32_t *qw, bool ov, cudaStream_t s) {
    const int M = p.a.M;
    return M == 1 ? launch_stream<1, LM, true, FMT>(p, qw, ov, s)
           : M <= 8 ? launch_stream<1, LM, false, FMT>(p, qw, ov, s)
                    : launch_stream<2, LM, false, FMT>(p, qw, ov, s);
}

template <bool LM>
int launch_stream_any(const StreamPlan &p, const uint32_t *qw, bool ov, cudaStream_t s) {
    const int fmt = fmt_class(p.a.f);
    return fmt == kFmtG64    ? launch_stream_f<LM, kFmtG64>(p, qw, ov, s)
           : fmt == kFmtS128 ? launch_stream_f<LM, kFmtS128>(p, qw, ov, s)
           : fmt == kFmtG32  ? launch_stream_f<LM, kFmtG32>(p, qw, ov, s)
                             : launch_stream_f<LM, kFmtAny>(p, qw, ov, s);
}

int gemv_impl(const uint16_t *x, const uint32_t *qw, const uint16_t *sc, const uint16_t *bi, uint16_t *y, int M,
              int N, int K, int group, unsigned flags, void *stream) {
    WFmt f;
    int st = check_common(x, qw, sc, bi, M, N, K, group, f);
    if (st != W4A16_OK) return st;
    if (!y) return W4_ERR_NULL;
    if (!aligned16(y)) return W4_ERR_ALIGN;
    if (flags & ~(unsigned)W4A16_OVERLAP_PREVIOUS) return W4_ERR_SHAPE;
    StreamPlan p;
    if (!plan_stream(p, M, N, K, f, false, 1)) return W4_ERR_SHAPE;
    p.a.x = x;
    p.a.sc = sc;
    p.a.bi = bi;
    p.a.y = y;
    p.a.ws = nullptr;
    const bool ov = (flags & W4A16_OVERLAP_PREVIOUS) != 0;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return launch_stream_any<false>(p, qw, ov, s);
}

int lmhead_impl(const uint16_t *x, const uint32_t *qw, const uint16_t *sc, const uint16_t *bi, int M, int N, int K,
                const WFmt &f, int k, int32_t *idx, float *val, uint64_t *ws, size_t ws_bytes, unsigned flags,
                void *stream) {
    StreamPlan p;
    if (!plan_stream(p, M, N, K, f, true, k)) return W4_ERR_SHAPE;
    const int G = p.grid;
    if ((long long)G > lm_max_blocks(N, k)) return W4_ERR_SHAPE;
    if (ws_bytes < (size_t)M * G * k * sizeof(uint64_t)) return W4_ERR_WORKSPACE;
    p.a.x = x;
    p.a.sc = sc;
    p.a.bi = bi;
    p.a.y = nullptr;
    p.a.ws = ws;
    const bool ov = (flags & W4A16_OVERLAP_PREVIOUS) != 0;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int st = launch_stream_any<true>(p, qw, ov, s);
    if (st != W4A16_OK) return st;
    // Pass 2 is launched as a programmatic dependent: its launch overlaps pass 1
    // and it waits (griddepcontrol.wait) for pass 1's results.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(M, 1, 1);
    cfg.blockDim = dim3(kPass2Threads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, lmhead_pass2, (const uint64_t *)ws, G, k, idx, val);
    return e == cudaSuccess ? W4A16_OK : W4_ERR_LAUNCH;
}

int lmhead_checks(const uint16_t *x, const uint32_t *qw, const uint16_t *sc, const uint16_t *bi, int M, int N, int K,
                  int group, int k, int32_t *idx, float *val, WFmt &f) {
    int st = check_common(x, qw, sc, bi, M, N, K, group, f);
    if (st != W4A16_OK) return st;
    if (!idx || !val) return W4_ERR_NULL;
    if (k < 1 || k > 64 || k > N || (long long)N * k > 16777216LL) return W4_ERR_SHAPE;
    if (!aligned16(idx) || !aligned16(val)) return W4_ERR_ALIGN;
    return W4A16_OK;
}

// Shared-memory layout of one sequence launch; false if it cannot fit.
// sc_max: the largest scale (and bias) bytes of a tile row block over the
// operations; xs_max: the most activation sums per row (groups, twice for
// group 32).
bool plan_seq(SeqParams &P, size_t &smem, int ng_max, size_t sc_max, int xs_max, int ntl_max) {
    const int M = P.M;
    // Partials of the 8 warps of each tile a CTA holds, and at least two
    // tiles' worth: a single tile split by K between the two teams keeps 16.
    if (ntl_max < 2) ntl_max = 2;
    P.w_bytes = (uint32_t)(kChunkGroups / kBoxGroups) * kBoxBytes;
    P.stage_bytes = (uint32_t)align_up((size_t)P.w_bytes + sc_max, 1024);
    const size_t fixed = align_up((size_t)ng_max * M * 128, 16) + align_up((size_t)xs_max * M * 4, 16) +
                         align_up((size_t)ntl_max * kSeqTeamWarps * kTileRows * M * 4, 16) + 16 * kMaxStages + 16 + 1024;
    if (fixed + 2 * (size_t)P.stage_bytes > (size_t)kMaxSmem) return false;
    P.stages = (int)min((size_t)kMaxStages, ((size_t)kMaxSmem - fixed) / P.stage_bytes);
    size_t off = (size_t)P.stages * P.stage_bytes;
    P.off_xf = (uint32_t)off;
    off = align_up(off + (size_t)ng_max * M * 128, 16);
    P.off_xsum = (uint32_t)off;
    off = align_up(off + (size_t)xs_max * M * 4, 16);
    P.off_red = (uint32_t)off;
    off = align_up(off + (size_t)ntl_max * kSeqTeamWarps * kTileRows * M * 4, 16);
    P.off_bar = (uint32_t)off;
    off += 16 * P.stages + 16;
    smem = off + 1024;
    return smem <= (size_t)kMaxSmem;
}

// Which activations of a launch's operations come from an earlier operation
// of the same launch: for operation c with wait_prev, the latest earlier
// operation whose output range overlaps x; when x lies inside that output,
// c reads its tagged copy (src[c] = that operation), otherwise it falls back to
// the completion counter (src[c] = -1).  tagged[i]: operation i's output is
// read this way.  Returns the tagged-copy bytes the launch needs.
size_t seq_sources(const w4_gemv_op *ops, int nops, int M, int *src, bool *tagged) {
    for (int i = 0; i < nops; ++i) {
        src[i] = -1;
        tagged[i] = false;
    }
    for (int c = 1; c < nops; ++c) {
        if (!ops[c].wait_prev) continue;
        const uintptr_t x0 = reinterpret_cast<uintptr_t>(ops[c].x);
        const uintptr_t x1 = x0 + (uintptr_t)M * ops[c].K * 2;
        for (int i = c - 1; i >= 0; --i) {
            const uintptr_t y0 = reinterpret_cast<uintptr_t>(ops[i].y);
            const uintptr_t y1 = y0 + (uintptr_t)M * ops[i].N * 2;
            if (x1 <= y0 || y1 <= x0) continue;  // disjoint
            if (x0 >= y0 && x1 <= y1 && (x0 - y0) % 2 == 0) {
                src[c] = i;
                tagged[i] = true;
            }
            break;
        }
    }
    size_t bytes = 0;
    for (int i = 0; i < nops; ++i)
        if (tagged[i]) bytes += align_up((size_t)M * ops[i].N * 4, 16);
    return bytes;
}

template <int FMT>
const void *seq_kernel_ptr(int M) {
    return M == 1 ? (const void *)seq_kernel<1, true, FMT>
           : M <= 8 ? (const void *)seq_kernel<1, false, FMT> : (const void *)seq_kernel<2, false, FMT>;
}

// Counter-wait settings of later launches (w4a16_testing_set_seq_wait).
std::atomic<unsigned long long> g_seq_wait_ns{kWaitNs};
std::atomic<unsigned> g_seq_target_bump{0u};

// Launch plans (tensor maps, tagged-exchange layout, shared-memory layout) of
// recent operation lists, so that a decode loop that passes the same list
// every token pays for planning and tensor-map encoding once.  An entry is
// reused only for an identical list (every field of every operation), the
// same rows M, workspace and device.
struct SeqPlan {
    int dev, nops, M;
    unsigned *ws;
    uint8_t *tagbuf;
    size_t tag_bytes;
    w4_gemv_op ops[kSeqMaxOps];
    SeqParams P;
    size_t smem;
    const void *kern;
    unsigned long long used;
};
constexpr int kSeqPlans = 8;

bool same_list(const SeqPlan &e, const w4_gemv_op *ops, int nops, int M, unsigned *ws, uint8_t *tagbuf,
               size_t tag_bytes, int dev) {
    if (e.nops != nops || e.M != M || e.ws != ws || e.tagbuf != tagbuf || e.tag_bytes != tag_bytes || e.dev != dev)
        return false;
    for (int i = 0; i < nops; ++i) {
        const w4_gemv_op &a = e.ops[i], &b = ops[i];
        if (a.x != b.x || a.qweight != b.qweight || a.scales != b.scales || a.biases != b.biases || a.y != b.y ||
            a.N != b.N || a.K != b.K || a.wait_prev != b.wait_prev || a.group != b.group)
            return false;
    }
    return true;
}

// Fills e.P, e.smem and e.kern for the list; a status other than W4A16_OK
// leaves the entry unusable.
int build_seq_plan(SeqPlan &e, const w4_gemv_op *ops, int nops, int M, unsigned *ws, uint8_t *tagbuf,
                   size_t tag_bytes) {
    static int src[kSeqMaxOps];
    static bool tagged[kSeqMaxOps];
    SeqParams &P = e.P;
    const int G = sm_count();
    // Tagged exchange when the workspace has room for it, else the counter.
    const bool use_tags = tagbuf && seq_sources(ops, nops, M, src, tagged) <= tag_bytes;
    uint32_t *yts[kSeqMaxOps];
    size_t toff = 0;
    for (int i = 0; i < nops; ++i) {
        yts[i] = nullptr;
        if (use_tags && tagged[i]) {
            yts[i] = reinterpret_cast<uint32_t *>(tagbuf + toff);
            toff += align_up((size_t)M * ops[i].N * 4, 16);
        }
    }
    int ng_max = 1, ntl_max = 1, xs_max = 1;
    size_t sc_max = 0;
    for (int i = 0; i < nops; ++i) {
        const w4_gemv_op &o = ops[i];
        SeqOp &d = P.ops[i];
        d.x = o.x;
        d.sc = o.scales;
        d.bi = o.biases;
        d.y = o.y;
        d.N = o.N;
        d.K = o.K;
        d.wait_prev = o.wait_prev;
        d.yt = yts[i];
        d.src = use_tags ? src[i] : -1;
        d.xt = d.src >= 0 ? yts[d.src] + (reinterpret_cast<const uint16_t *>(o.x) - ops[d.src].y) : nullptr;
        const int nq = o.K / 256;
        d.cq = min(kChunkGroups / kBoxGroups, nq);
        ng_max = max(ng_max, o.K / kGroup);
        // Checked by the caller.
        make_fmt(d.f, o.K, o.group ? o.group : kGroup, o.biases == nullptr);
        sc_max = std::max(sc_max, (size_t)(d.f.sym ? 32 : 64) * d.f.ngs);
        xs_max = max(xs_max, (o.K / kGroup) * (d.f.gs == 0 ? 2 : 1));
        ntl_max = max(ntl_max, ((o.N + kTileRows - 1) / kTileRows + G - 1) / G);
        const uint64_t KW = (uint64_t)o.K / 8;
        if (!make_map_3d(&P.maps[i], CU_TENSOR_MAP_DATA_TYPE_UINT32, o.qweight, 32, (uint64_t)o.N, (uint64_t)nq,
                         KW * 4, 128, 32, kTileRows, (uint32_t)d.cq, CU_TENSOR_MAP_SWIZZLE_128B))
            return W4_ERR_DEVICE;
    }
    P.nops = nops;
    P.M = M;
    P.ws = ws;
    P.publish = 0;
    for (int i = 1; i < nops; ++i)
        if (P.ops[i].wait_prev && !P.ops[i].xt) P.publish = 1;
    if (!plan_seq(P, e.smem, ng_max, sc_max, xs_max, ntl_max)) return W4_ERR_SHAPE;
    const int fmt = fmt_class(P.ops[0].f);  // the same for every operation of a launch
    e.kern = fmt == kFmtG64    ? seq_kernel_ptr<kFmtG64>(M)
             : fmt == kFmtS128 ? seq_kernel_ptr<kFmtS128>(M)
             : fmt == kFmtG32  ? seq_kernel_ptr<kFmtG32>(M)
                               : seq_kernel_ptr<kFmtAny>(M);
    return W4A16_OK;
}

int seq_launch(const w4_gemv_op *ops, int nops, int M, unsigned *ws, uint8_t *tagbuf, size_t tag_bytes,
               cudaStream_t st) {
    static SeqPlan plans[kSeqPlans];  // large: kept off the stack
    static unsigned long long clock = 0;
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return W4_ERR_DEVICE;
    SeqPlan *e = nullptr;
    for (int i = 0; i < kSeqPlans && !e; ++i)
        if (plans[i].nops > 0 && same_list(plans[i], ops, nops, M, ws, tagbuf, tag_bytes, dev)) e = &plans[i];
    if (!e) {
        e = &plans[0];  // least recently used (or empty) entry
        for (int i = 1; i < kSeqPlans; ++i)
            if (plans[i].used < e->used) e = &plans[i];
        e->nops = 0;
        const int bs = build_seq_plan(*e, ops, nops, M, ws, tagbuf, tag_bytes);
        if (bs != W4A16_OK) return bs;
        e->dev = dev;
        e->nops = nops;
        e->M = M;
        e->ws = ws;
        e->tagbuf = tagbuf;
        e->tag_bytes = tag_bytes;
        for (int i = 0; i < nops; ++i) e->ops[i] = ops[i];
    }
    e->used = ++clock;
    SeqParams &P = e->P;
    P.wait_ns = g_seq_wait_ns.load();
    P.target_bump = g_seq_target_bump.load();
    const size_t smem = e->smem;
    const void *kern = e->kern;
    if (!ensure_smem(kern, smem)) return W4_ERR_LAUNCH;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(sm_count(), 1, 1);
    cfg.blockDim = dim3(kSeqThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;  // every CTA resident: the waits cannot starve
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void *args[] = {&P};
    const cudaError_t err = cudaLaunchKernelExC(&cfg, kern, args);
    if (err != cudaSuccess) {
        cudaGetLastError();
        return W4_ERR_LAUNCH;
    }
    return W4A16_OK;
}

}  // namespace
}  // namespace w4a16

using namespace w4a16;

extern "C" int w4_gemv(const uint16_t *x, const uint32_t *qweight, const uint16_t *scales, const uint16_t *biases,
                       uint16_t *y, int M, int N, int K, int group, void *stream) {
    return gemv_impl(x, qweight, scales, biases, y, M, N, K, group, 0u, stream);
}

extern "C" int w4_gemv_ex(const uint16_t *x, const uint32_t *qweight, const uint16_t *scales, const uint16_t *biases,
                          uint16_t *y, int M, int N, int K, int group, unsigned flags, void *stream) {
    return gemv_impl(x, qweight, scales, biases, y, M, N, K, group, flags, stream);
}

extern "C" size_t lm_head_workspace_bytes(int M, int N, int k) {
    if (M < 1 || M > 16 || N < 1 || k < 1 || k > 64 || k > N) return 0;
    if ((long long)N * k > 16777216LL) return 0;
    return (size_t)M * (size_t)lm_max_blocks(N, k) * (size_t)k * sizeof(uint64_t);
}

extern "C" int lm_head_argmax_topk(const uint16_t *x, const uint32_t *qweight, const uint16_t *scales,
                                   const uint16_t *biases, int M, int N, int K, int group, int k, int32_t *idx,
                                   float *val, void *workspace, size_t workspace_bytes, void *stream) {
    WFmt f;
    int st = lmhead_checks(x, qweight, scales, biases, M, N, K, group, k, idx, val, f);
    if (st != W4A16_OK) return st;
    if (!workspace || workspace_bytes < lm_head_workspace_bytes(M, N, k)) return W4_ERR_WORKSPACE;
    if (!aligned16(workspace)) return W4_ERR_ALIGN;
    return lmhead_impl(x, qweight, scales, biases, M, N, K, f, k, idx, val,
                       reinterpret_cast<uint64_t *>(workspace), workspace_bytes, 0u, stream);
}

extern "C" int lm_head_argmax_topk_ex(const uint16_t *x, const uint32_t *qweight, const uint16_t *scales,
                                      const uint16_t *biases, int M, int N, int K, int group, int k, int32_t *idx,
                                      float *val, void *workspace, size_t workspace_bytes, unsigned flags,
                                      void *stream) {
    WFmt f;
    int st = lmhead_checks(x, qweight, scales, biases, M, N, K, group, k, idx, val, f);
    if (st != W4A16_OK) return st;
    if (flags & ~(unsigned)W4A16_OVERLAP_PREVIOUS) return W4_ERR_SHAPE;
    if (!workspace || workspace_bytes < lm_head_workspace_bytes(M, N, k)) return W4_ERR_WORKSPACE;
    if (!aligned16(workspace)) return W4_ERR_ALIGN;
    return lmhead_impl(x, qweight, scales, biases, M, N, K, f, k, idx, val,
                       reinterpret_cast<uint64_t *>(workspace), workspace_bytes, flags, stream);
}

// Scale-layout class of an operation (its arguments need not be valid yet).
static int seq_op_class(const w4_gemv_op &o) {
    const int group = o.group ? o.group : kGroup;
    if (group == 32) return kFmtG32;
    if (group == kGroup && o.biases) return kFmtG64;
    if (group == 2 * kGroup && !o.biases) return kFmtS128;
    return kFmtAny;
}

// Operations of the next launch of a list: up to kSeqMaxOps of one scale-layout
// class (one kernel variant per launch).
static int seq_launch_ops(const w4_gemv_op *ops, int nops) {
    const int c = seq_op_class(ops[0]);
    int n = 1;
    while (n < nops && n < kSeqMaxOps && seq_op_class(ops[n]) == c) ++n;
    return n;
}

extern "C" size_t w4_gemv_seq_workspace_bytes(void) { return kSeqCounterBytes; }

extern "C" int w4a16_testing_set_seq_wait(unsigned long long wait_ns, unsigned target_bump) {
    if (wait_ns > kWaitNs) return W4_ERR_SHAPE;
    g_seq_wait_ns.store(wait_ns ? wait_ns : kWaitNs);
    g_seq_target_bump.store(target_bump);
    return W4A16_OK;
}

extern "C" size_t w4_gemv_seq_workspace_bytes_ex(const w4_gemv_op *ops, int nops, int M) {
    if (!ops || nops < 1 || M < 1 || M > 16) return kSeqCounterBytes;
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    static int src[kSeqMaxOps];
    static bool tagged[kSeqMaxOps];
    size_t most = 0;
    for (int first = 0, n = 0; first < nops; first += n) {
        n = seq_launch_ops(ops + first, nops - first);
        most = std::max(most, seq_sources(ops + first, n, M, src, tagged));
    }
    return kSeqCounterBytes + most;
}

extern "C" int w4_gemv_seq(const w4_gemv_op *ops, int nops, int M, void *workspace, size_t workspace_bytes,
                           unsigned flags, void *stream) {
    if (!ops || !workspace) return ops ? W4_ERR_WORKSPACE : W4_ERR_NULL;
    if (workspace_bytes < w4_gemv_seq_workspace_bytes()) return W4_ERR_WORKSPACE;
    if (!aligned16(workspace)) return W4_ERR_ALIGN;
    if (nops < 1 || M < 1 || M > 16 || flags != 0) return W4_ERR_SHAPE;
    for (int i = 0; i < nops; ++i) {
        const w4_gemv_op &o = ops[i];
        WFmt f;
        if (o.group < 0) return W4_ERR_GROUP;
        int st = check_common(o.x, o.qweight, o.scales, o.biases, M, o.N, o.K, o.group ? o.group : kGroup, f);
        if (st != W4A16_OK) return st;
        if (!o.y) return W4_ERR_NULL;
        if (!aligned16(o.y)) return W4_ERR_ALIGN;
        if (o.K % 256 != 0) return W4_ERR_SHAPE;  // whole 128-byte quads per row
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    for (int first = 0, n = 0; first < nops; first += n) {
        n = seq_launch_ops(ops + first, nops - first);
        uint8_t *ws8 = reinterpret_cast<uint8_t *>(workspace);
        const int st = seq_launch(ops + first, n, M, reinterpret_cast<unsigned *>(workspace),
                                  workspace_bytes > kSeqCounterBytes ? ws8 + kSeqCounterBytes : nullptr,
                                  workspace_bytes - kSeqCounterBytes, s);
        if (st != W4A16_OK) return st;
    }
    return W4A16_OK;
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

// Unique id of the current CUDA context (cuCtxGetId: never reused within a
// process), or 0 if the driver does not provide it.
unsigned long long current_context_id() {
    typedef CUresult (*GetCurrentFn)(CUcontext *);
    typedef CUresult (*GetIdFn)(CUcontext, unsigned long long *);
    static GetCurrentFn get_current = nullptr;
    static GetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<GetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<GetIdFn>(p);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of g_lm_scratch in the current device's context.  The
// host-side name is only a stand-in; the address is looked up with the device
// current and cached per device together with the id of the context it
// belongs to, so a new primary context (after cudaDeviceReset) gets a fresh
// lookup.  Without context ids the address is looked up on every call.
void *noalloc_scratch() {
    static std::mutex mu;
    static void *addr[64] = {nullptr};
    static unsigned long long ctx_of[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    const unsigned long long ctx = current_context_id();
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev] || ctx == 0 || ctx_of[dev] != ctx) {
        // (The lookup also makes the device's primary context current.)
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_lm_scratch) != cudaSuccess) {
            cudaGetLastError();
            addr[dev] = nullptr;
            return nullptr;
        }
        addr[dev] = p;
        ctx_of[dev] = ctx ? ctx : current_context_id();
    }
    return addr[dev];
}

}  // namespace
}  // namespace w4a16

extern "C" int lm_head_argmax_topk_noalloc(const uint16_t *x, const uint32_t *qweight, const uint16_t *scales,
                                           const uint16_t *biases, int M, int N, int K, int group, int k,
                                           int32_t *idx, float *val, void *stream) {
    WFmt f;
    int st = lmhead_checks(x, qweight, scales, biases, M, N, K, group, k, idx, val, f);
    if (st != W4A16_OK) return st;
    const size_t need = lm_head_workspace_bytes(M, N, k);
    if (need == 0 || need > kNoAllocScratchBytes) return W4_ERR_WORKSPACE;
    void *scratch = noalloc_scratch();
    if (!scratch) return W4_ERR_DEVICE;
    return lmhead_impl(x, qweight, scales, biases, M, N, K, f, k, idx, val,
                       reinterpret_cast<uint64_t *>(scratch), kNoAllocScratchBytes, 0u, stream);
}
