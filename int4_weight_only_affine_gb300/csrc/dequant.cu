// w4_dequant_f16: dequantise once into the transposed half scratch.
//
// "The inference engine - Mojo 1.0 on Metal", "Crossing Mojo 1.0": prefill
// dequantises each weight once into a transposed half-precision scratch and
// then runs a half-precision GEMM on it.
//
// w16[k][n] = RNE_binary16(scale[n][k/G] * q[n][k] + bias[n][k/G]), or
// RNE_binary16(scale[n][k/G] * (q[n][k] - 8)) for symmetric codes.
// The code is made an exact binary16 (1024 + q via the exponent trick, then an
// exact subtraction of 1024, or of 1032 for q - 8) and one binary16 fused
// multiply-add (a multiply for symmetric codes) rounds the exact value once,
// to nearest even: the correctly rounded value.
//
// The kernels are HBM bound (0.5625 B read + 2 B written per weight).
//
// dequant_tma_kernel (N % 8 == 0): persistent CTAs, two per SM, walk tiles of
// 64 rows x 256 k.  Thread 0 brings each tile's codes in with one TMA copy
// (128-byte swizzle, four tiles in flight) and writes each finished tile out
// with one TMA store of the transposed [256 k][64 n] binary16 block (two
// output buffers, the store of one overlapping the conversion of the next).
// Lane l converts rows 2l and 2l+1 as (row, row+1) half pairs over the
// 32 k of its 16-byte chunk; the chunk index varies with the lane so that the
// swizzled reads hit every bank, and every output row is 128 bytes, so the
// pair stores are conflict-free.  Scales and biases are loaded into
// registers two tiles ahead of their use.
//
// dequant_kernel (any N): tiles of 64 rows x 64 k: threads read the codes of
// two adjacent rows, dequantise them as (row n, row n+1) half pairs,
// transpose through padded shared memory, and write 128-byte segments of 64
// consecutive n for each k.
#include <type_traits>

#include "common.cuh"

namespace w4a16 {
namespace {

constexpr int kTileN = 64;              // rows of W per tile (= n columns of w16)
constexpr int kPairs = kTileN / 2;      // 32-bit (n, n+1) pairs per k row
constexpr int kStride = kPairs + 1;     // padded shared-memory row (words)
constexpr int kThreads = 256;

// The half pairs (w(row a), w(row b)) of the eight codes of words A (row a)
// and B (row b) with scales s2 and biases b2; symmetric: bias-free, code
// q - 8.  koff: 1024 (affine) or 1032 (symmetric) in both halves.
template <bool SYM>
__device__ __forceinline__ void dequant_word_pair(uint32_t A, uint32_t B, __half2 s2, __half2 b2, __half2 koff,
                                                  uint32_t (&o)[8]) {
    // (row a, row b) pairs of codes 0..3 and 4..7 of this word.
    const uint32_t lo = __byte_perm(A, B, 0x5410);
    const uint32_t hi = __byte_perm(A, B, 0x7632);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const uint32_t src = e < 4 ? lo : hi;
        const uint32_t v = ((src >> (4 * (e & 3))) & 0x000F000Fu) | 0x64006400u;  // 1024 + q
        const __half2 q2 = __hsub2(*reinterpret_cast<const __half2 *>(&v), koff);  // exact q (or q - 8)
        const __half2 w2 = SYM ? __hmul2(q2, s2) : __hfma2(q2, s2, b2);           // one rounding
        o[e] = *reinterpret_cast<const uint32_t *>(&w2);
    }
}

__global__ void __launch_bounds__(kThreads)
    dequant_kernel(const uint32_t *__restrict__ qw, const uint16_t *__restrict__ sc,
                   const uint16_t *__restrict__ bi, uint16_t *__restrict__ w16, int N, int K,
                   long long ntiles, int tiles_n, WFmt f) {
    __shared__ uint32_t tile[kGroup * kStride];
    // Warp w covers 8 row pairs x 4 words: shared-memory stores (bank
    // 8*word + i + pair, mod 32) are conflict free.
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int pair = (warp & 3) * 8 + (lane >> 2);  // 0..31
    const int word = (warp >> 2) * 4 + (lane & 3);  // word of the group, k = 8*word .. 8*word+7
    const bool vec_ok = (N % 8) == 0;

    for (long long t = blockIdx.x; t < ntiles; t += gridDim.x) {
        const int G = (int)(t / tiles_n);
        const int n0 = (int)(t % tiles_n) * kTileN;
        const int na = min(n0 + 2 * pair, N - 1);
        const int nb = min(n0 + 2 * pair + 1, N - 1);
        const uint32_t A = __ldg(qw + (size_t)na * (K / 8) + (size_t)G * kWordsPerGroup + word);
        const uint32_t B = __ldg(qw + (size_t)nb * (K / 8) + (size_t)G * kWordsPerGroup + word);
        const int gi = (G * kGroup + 8 * word) >> (f.gs + 5);  // quantisation group of the word
        const uint16_t sa = ld_nc_u16(sc + (size_t)na * f.ngs + gi), sb = ld_nc_u16(sc + (size_t)nb * f.ngs + gi);
        const __half2 s2 = __halves2half2(__ushort_as_half(sa), __ushort_as_half(sb));
        uint32_t o[8];
        if (f.sym) {
            dequant_word_pair<true>(A, B, s2, s2, __float2half2_rn(1032.f), o);
        } else {
            const uint16_t ba = ld_nc_u16(bi + (size_t)na * f.ngs + gi), bb = ld_nc_u16(bi + (size_t)nb * f.ngs + gi);
            const __half2 b2 = __halves2half2(__ushort_as_half(ba), __ushort_as_half(bb));
            dequant_word_pair<false>(A, B, s2, b2, __float2half2_rn(1024.f), o);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) tile[(8 * word + i) * kStride + pair] = o[i];
        __syncthreads();
        // 64 k rows x 32 words; each thread writes 4 words (8 n) per pass.
#pragma unroll
        for (int pass = 0; pass < 2; ++pass) {
            const int r = pass * 32 + (threadIdx.x >> 3);
            const int cw = (threadIdx.x & 7) * 4;
            const size_t off = (size_t)(G * kGroup + r) * N + n0 + 2 * cw;
            const uint32_t *srow = tile + r * kStride + cw;
            if (vec_ok && n0 + 2 * cw + 8 <= N) {
                uint4 v = make_uint4(srow[0], srow[1], srow[2], srow[3]);
                *reinterpret_cast<uint4 *>(w16 + off) = v;
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int n = n0 + 2 * (cw + e);
                    if (n < N) w16[off + 2 * e] = (uint16_t)(srow[e] & 0xFFFFu);
                    if (n + 1 < N) w16[off + 2 * e + 1] = (uint16_t)(srow[e] >> 16);
                }
            }
        }
        __syncthreads();
    }
}

constexpr int kTmaRows = 64;                       // rows of W per tile (= n columns of w16)
constexpr int kTmaK = 256;                         // k per tile (4 groups, 32 words per row)
constexpr int kCodeBytes = kTmaRows * kTmaK / 2;   // 8 KB
constexpr int kOutBytes = kTmaK * kTmaRows * 2;    // 32 KB
constexpr int kCodeStages = 4;                    // code tiles in flight per CTA
// Scale staging: ANY keeps a pair (the two 32-k chunks) per row and 64-k block.
template <bool ANY>
constexpr int tma_smem() {
    return kCodeStages * kCodeBytes + 2 * kOutBytes + 2 * 2 * kTmaRows * 4 * (ANY ? 4 : 2) + 8 * kCodeStages;
}

// ANY: any scale layout (f); otherwise group-64 affine (one scale and one
// bias per 64-k block).
template <bool ANY>
__global__ void __launch_bounds__(kThreads, 2)
    dequant_tma_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_w,
                       const uint16_t *__restrict__ sc, const uint16_t *__restrict__ bi, int N, int K, int tiles_n,
                       int ntiles, WFmt f) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = (uint32_t)__cvta_generic_to_shared(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *sb = smem_raw + (base - raw);
    constexpr int kOutOff = kCodeStages * kCodeBytes;
    const uint32_t codes0 = base, out0 = base + kOutOff;
    // Scales and biases of each row and 64-k block of a tile, [2][64][4]:
    // group 64 one binary16 each; ANY the pair of its 32-k chunks (low half
    // first).
    using SW = typename std::conditional<ANY, uint32_t, uint16_t>::type;
    SW *scl = reinterpret_cast<SW *>(sb + kOutOff + 2 * kOutBytes);
    SW *bia = scl + 2 * kTmaRows * 4;
    const uint32_t bar0 = base + kOutOff + 2 * kOutBytes + 2 * 2 * kTmaRows * 4 * (int)sizeof(SW);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = gridDim.x;
    // Launched with W4A16_OVERLAP_PREVIOUS the caller guarantees independence
    // from the previous and the next kernel: release the next one at once
    // (without the attribute this is ordinary stream order).
    pdl_launch_dependents();
    auto tile_n0 = [&](int t) { return (t % tiles_n) * kTmaRows; };
    auto tile_k0 = [&](int t) { return (t / tiles_n) * kTmaK; };
    // Thread tid stages the scales and biases of row tid/4, 64-k block tid%4
    // of a tile.
    auto load_sb = [&](int t, SW &s, SW &b) {
        const int n = min(tile_n0(t) + tid / 4, N - 1);
        if (!ANY) {
            const int g = min(tile_k0(t) / kGroup + (tid & 3), f.ngs - 1);
            s = ld_nc_u16(sc + (size_t)n * f.ngs + g);
            b = ld_nc_u16(bi + (size_t)n * f.ngs + g);
            return;
        }
        const int c0 = min(tile_k0(t) + 64 * (tid & 3), K - 64) >> 5;  // first 32-k chunk along K
        const int g0 = c0 >> f.gs, g1 = (c0 + 1) >> f.gs;
        const uint16_t *rs = sc + (size_t)n * f.ngs;
        s = (SW)((uint32_t)ld_nc_u16(rs + g0) | ((uint32_t)ld_nc_u16(rs + g1) << 16));
        b = 0u;
        if (!f.sym) {
            const uint16_t *rb = bi + (size_t)n * f.ngs;
            b = (SW)((uint32_t)ld_nc_u16(rb + g0) | ((uint32_t)ld_nc_u16(rb + g1) << 16));
        }
    };

    if (tid == 0) {
        for (int i = 0; i < kCodeStages; ++i) mbar_init(bar0 + 8 * i, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        for (int i = 0; i < kCodeStages; ++i) {
            const int t = blockIdx.x + i * G;
            if (t < ntiles) {
                mbar_expect_tx(bar0 + 8 * i, kCodeBytes);
                tma_load_2d(codes0 + i * kCodeBytes, &map_q, tile_k0(t) / 8, tile_n0(t), bar0 + 8 * i);
            }
        }
    }
    // Scales: tile 0's into shared memory now; tile i+1's are in registers
    // (loaded two tiles ahead) and reach shared memory at the end of tile i.
    SW ps0 = 0, pb0 = 0, ps1 = 0, pb1 = 0;  // register sets for even / odd tiles
    if (blockIdx.x < ntiles) {
        SW s, b;
        load_sb(blockIdx.x, s, b);
        scl[tid] = s;
        bia[tid] = b;
    }
    if (blockIdx.x + G < ntiles) load_sb(blockIdx.x + G, ps1, pb1);
    __syncthreads();

    // Lane l: rows 2l, 2l+1; 16-byte chunk c of the 128-byte row (k = 32c..32c+31).
    const int c = (warp + (lane >> 2)) & 7;
    const int rowa = 2 * lane, rowb = 2 * lane + 1;
    const uint32_t offa = rowa * 128 + ((c ^ (rowa & 7)) << 4);
    const uint32_t offb = rowb * 128 + ((c ^ (rowb & 7)) << 4);
    const __half2 koff = __float2half2_rn(ANY && f.sym ? 1032.f : 1024.f);
    bool ok = true;
    int waited = 0;  // tiles whose codes this thread has waited for
    for (int i = 0;; ++i) {
        const int t = blockIdx.x + i * G;
        if (t >= ntiles) break;
        const int st = i & 1;              // output and scale buffer
        const int cst = i % kCodeStages;   // code buffer
        const int tn = t + G;
        if (t + 2 * G < ntiles) {  // scales two tiles ahead, into this tile's register set
            if (st == 0)
                load_sb(t + 2 * G, ps0, pb0);
            else
                load_sb(t + 2 * G, ps1, pb1);
        }
        if (ok) {
            ok = mbar_wait(bar0 + 8 * cst, (i / kCodeStages) & 1);
            if (ok) waited = i + 1;
        }
        if (tid == 0) bulk_wait_group_read<1>();  // the store that last used this output buffer has read it
        __syncthreads();
        if (ok) {
            const uint8_t *cs = sb + cst * kCodeBytes;
            const uint4 A = *reinterpret_cast<const uint4 *>(cs + offa);
            const uint4 B = *reinterpret_cast<const uint4 *>(cs + offb);
            // Scale and bias of chunk c: block c/2 of the row's set (ANY: half c%2).
            const int sh = 16 * (c & 1), wi = c >> 1;
            auto pair = [&](const SW *arr) {
                const uint32_t va = arr[st * 256 + rowa * 4 + wi], vb = arr[st * 256 + rowb * 4 + wi];
                const uint32_t p = ANY ? __byte_perm(va >> sh, vb >> sh, 0x5410) : __byte_perm(va, vb, 0x5410);
                return *reinterpret_cast<const __half2 *>(&p);
            };
            const __half2 s2 = pair(scl);
            uint32_t *out = reinterpret_cast<uint32_t *>(sb + kOutOff + st * kOutBytes);
            const uint32_t wa[4] = {A.x, A.y, A.z, A.w}, wb[4] = {B.x, B.y, B.z, B.w};
            if (ANY && f.sym) {
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    uint32_t o[8];
                    dequant_word_pair<true>(wa[w], wb[w], s2, s2, koff, o);
#pragma unroll
                    for (int e = 0; e < 8; ++e) out[(32 * c + 8 * w + e) * (kTmaRows / 2) + lane] = o[e];
                }
            } else {
                const __half2 b2 = pair(bia);
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    uint32_t o[8];
                    dequant_word_pair<false>(wa[w], wb[w], s2, b2, koff, o);
#pragma unroll
                    for (int e = 0; e < 8; ++e) out[(32 * c + 8 * w + e) * (kTmaRows / 2) + lane] = o[e];
                }
            }
        }
        fence_proxy_async_smem();  // the tile's generic writes before the TMA store reads them
        __syncthreads();
        if (tid == 0) {
            if (ok) {
                tma_store_2d(&map_w, out0 + st * kOutBytes, tile_n0(t), tile_k0(t));
                bulk_commit_group();
            }
            const int t2 = t + kCodeStages * G;  // refill this code buffer
            if (ok && t2 < ntiles) {
                mbar_expect_tx(bar0 + 8 * cst, kCodeBytes);
                tma_load_2d(codes0 + cst * kCodeBytes, &map_q, tile_k0(t2) / 8, tile_n0(t2), bar0 + 8 * cst);
            }
        }
        if (tn < ntiles) {
            scl[(st ^ 1) * 256 + tid] = st ? ps0 : ps1;
            bia[(st ^ 1) * 256 + tid] = st ? pb0 : pb1;
        }
    }
    if (tid == 0) {
        // After an expired wait: the code copies issued for tiles not waited
        // for still land before the CTA exits (bounded waits).
        for (int i = waited; i < waited + kCodeStages; ++i)
            if (blockIdx.x + i * G < ntiles) mbar_wait(bar0 + 8 * (i % kCodeStages), (i / kCodeStages) & 1);
        bulk_wait_group<0>();  // every store has landed before the CTA exits
    }
}

}  // namespace

// Reads and clears this translation unit's expired-wait record.
int dequant_wait_flag() {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_wait_expired, sizeof(int)) != cudaSuccess) return -1;
    if (v) {
        const int zero = 0;
        cudaMemcpyToSymbol(g_wait_expired, &zero, sizeof(int));
    }
    return v;
}
}  // namespace w4a16

using namespace w4a16;

static int dequant_impl(const uint32_t *qweight, const uint16_t *scales, const uint16_t *biases, uint16_t *w16,
                        int N, int K, int group, unsigned flags, void *stream) {
    if (!qweight || !scales || !w16) return W4_ERR_NULL;
    if (N < 1 || K < kGroup || K % kGroup != 0) return W4_ERR_SHAPE;
    WFmt f;
    if (!make_fmt(f, K, group, biases == nullptr)) return W4_ERR_GROUP;
    if (!aligned16(qweight) || !aligned16(scales) || (biases && !aligned16(biases)) || !aligned16(w16))
        return W4_ERR_ALIGN;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (N % 8 == 0) {
        // w16 rows are 16-byte multiples: tensor copies both ways.
        CUtensorMap mq, mw;
        const uint64_t KW = (uint64_t)K / 8;
        if (!make_map_2d(&mq, CU_TENSOR_MAP_DATA_TYPE_UINT32, qweight, KW, (uint64_t)N, KW * 4, 32, kTmaRows,
                         CU_TENSOR_MAP_SWIZZLE_128B) ||
            !make_map_2d(&mw, CU_TENSOR_MAP_DATA_TYPE_UINT16, w16, (uint64_t)N, (uint64_t)K, (uint64_t)N * 2,
                         kTmaRows, kTmaK, CU_TENSOR_MAP_SWIZZLE_NONE))
            return W4_ERR_DEVICE;
        const int tiles_n = (N + kTmaRows - 1) / kTmaRows;
        const long long ntiles = (long long)tiles_n * ((K + kTmaK - 1) / kTmaK);
        if (ntiles > 0x7fffffffLL) return W4_ERR_SHAPE;
        const bool any = !(f.gs == 1 && !f.sym);
        auto kern = any ? dequant_tma_kernel<true> : dequant_tma_kernel<false>;
        const int smem = (any ? tma_smem<true>() : tma_smem<false>()) + 1024;
        if (!set_smem_once(reinterpret_cast<const void *>(kern), smem)) return W4_ERR_LAUNCH;
        long long grid = (long long)sm_count() * 2;
        if (grid > ntiles) grid = ntiles;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)grid, 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = (flags & W4A16_OVERLAP_PREVIOUS) ? 1 : 0;
        const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, mq, mw, scales, biases, N, K, tiles_n, (int)ntiles, f);
        return e == cudaSuccess ? W4A16_OK : W4_ERR_LAUNCH;
    }
    const int tiles_n = (N + kTileN - 1) / kTileN;
    const long long ntiles = (long long)tiles_n * (K / kGroup);
    long long grid = (long long)sm_count() * 8;
    if (grid > ntiles) grid = ntiles;
    dequant_kernel<<<(unsigned)grid, kThreads, 0, st>>>(qweight, scales, biases, w16, N, K, ntiles, tiles_n, f);
    return launch_status();
}

extern "C" int w4_dequant_f16(const uint32_t *qweight, const uint16_t *scales, const uint16_t *biases,
                              uint16_t *w16, int N, int K, int group, void *stream) {
    return dequant_impl(qweight, scales, biases, w16, N, K, group, 0u, stream);
}

extern "C" int w4_dequant_f16_ex(const uint32_t *qweight, const uint16_t *scales, const uint16_t *biases,
                                 uint16_t *w16, int N, int K, int group, unsigned flags, void *stream) {
    if (flags & ~(unsigned)W4A16_OVERLAP_PREVIOUS) return W4_ERR_SHAPE;
    return dequant_impl(qweight, scales, biases, w16, N, K, group, flags, stream);
}
