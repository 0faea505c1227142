// w4_dequant_f16: dequantise once into the transposed half scratch.
//
// "The inference engine - Mojo 1.0 on Metal", "Crossing Mojo 1.0": prefill
// dequantises each weight once into a transposed half-precision scratch and
// then runs a half-precision GEMM on it.
//
// w16[k][n] = RNE_binary16(scale[n][k/64] * q[n][k] + bias[n][k/64]).
// The code is made an exact binary16 (1024 + q via the exponent trick, then an
// exact subtraction of 1024) and one binary16 fused multiply-add rounds the
// exact scale*q + bias once, to nearest even: the correctly rounded value.
//
// The kernel is HBM bound (0.5625 B read + 2 B written per weight).  A CTA
// handles tiles of 64 rows x 64 k: threads read the codes of two adjacent rows
// (16-byte row segments; the two warps covering a 32-byte group share it in L1), dequantise them as (row n, row n+1) half
// pairs, transpose through padded shared memory, and write 128-byte segments
// of 64 consecutive n for each k.
#include "common.cuh"

namespace w4a16 {
namespace {

constexpr int kTileN = 64;              // rows of W per tile (= n columns of w16)
constexpr int kPairs = kTileN / 2;      // 32-bit (n, n+1) pairs per k row
constexpr int kStride = kPairs + 1;     // padded shared-memory row (words)
constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads)
    dequant_kernel(const uint32_t *__restrict__ qw, const uint16_t *__restrict__ sc,
                   const uint16_t *__restrict__ bi, uint16_t *__restrict__ w16, int N, int K,
                   long long ntiles, int tiles_n) {
    __shared__ uint32_t tile[kGroup * kStride];
    const int ng = K / kGroup;
    // Warp w covers 8 row pairs x 4 words: shared-memory stores (bank
    // 8*word + i + pair, mod 32) are conflict free.
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int pair = (warp & 3) * 8 + (lane >> 2);  // 0..31
    const int word = (warp >> 2) * 4 + (lane & 3);  // word of the group, k = 8*word .. 8*word+7
    const bool vec_ok = (N % 8) == 0;
    const __half2 k1024 = __float2half2_rn(1024.f);

    for (long long t = blockIdx.x; t < ntiles; t += gridDim.x) {
        const int G = (int)(t / tiles_n);
        const int n0 = (int)(t % tiles_n) * kTileN;
        const int na = min(n0 + 2 * pair, N - 1);
        const int nb = min(n0 + 2 * pair + 1, N - 1);
        const uint32_t A = __ldg(qw + (size_t)na * (K / 8) + (size_t)G * kWordsPerGroup + word);
        const uint32_t B = __ldg(qw + (size_t)nb * (K / 8) + (size_t)G * kWordsPerGroup + word);
        const uint16_t sa = ld_nc_u16(sc + (size_t)na * ng + G), sb = ld_nc_u16(sc + (size_t)nb * ng + G);
        const uint16_t ba = ld_nc_u16(bi + (size_t)na * ng + G), bb = ld_nc_u16(bi + (size_t)nb * ng + G);
        const __half2 s2 = __halves2half2(__ushort_as_half(sa), __ushort_as_half(sb));
        const __half2 b2 = __halves2half2(__ushort_as_half(ba), __ushort_as_half(bb));
        // (row n, row n+1) pairs of codes 0..3 and 4..7 of this word.
        const uint32_t lo = __byte_perm(A, B, 0x5410);
        const uint32_t hi = __byte_perm(A, B, 0x7632);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t src = (i < 4) ? lo : hi;
            const uint32_t v = ((src >> (4 * (i & 3))) & 0x000F000Fu) | 0x64006400u;  // 1024 + q
            __half2 q2 = __hsub2(*reinterpret_cast<const __half2 *>(&v), k1024);   // exact q
            __half2 w2 = __hfma2(q2, s2, b2);                                     // one rounding
            tile[(8 * word + i) * kStride + pair] = *reinterpret_cast<uint32_t *>(&w2);
        }
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

}  // namespace
}  // namespace w4a16

using namespace w4a16;

extern "C" int w4_dequant_f16(const uint32_t *qweight, const uint16_t *scales, const uint16_t *biases,
                              uint16_t *w16, int N, int K, int group, void *stream) {
    if (!qweight || !scales || !biases || !w16) return W4_ERR_NULL;
    if (group != kGroup) return W4_ERR_GROUP;
    if (N < 1 || K < kGroup || K % kGroup != 0) return W4_ERR_SHAPE;
    if (!aligned16(qweight) || !aligned16(scales) || !aligned16(biases) || !aligned16(w16))
        return W4_ERR_ALIGN;
    const int tiles_n = (N + kTileN - 1) / kTileN;
    const long long ntiles = (long long)tiles_n * (K / kGroup);
    long long grid = (long long)sm_count() * 8;
    if (grid > ntiles) grid = ntiles;
    dequant_kernel<<<(unsigned)grid, kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        qweight, scales, biases, w16, N, K, ntiles, tiles_n);
    return launch_status();
}
