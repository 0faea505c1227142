// Consumer-side arithmetic of the W4A16 GEMV kernels: activation staging in
// MMA fragment order and the per-group tensor-core dot products with the
// affine step folded in.  Shared by the streaming and projection-list kernels.
//
// Here a "group" is a 64-k block of codes (8 words of a row), the unit the
// kernels step by.  The quantisation group (WFmt) may span several blocks
// (group 128, 256, ...: the blocks share a scale) or half of one (group 32:
// the G32 variants keep the two halves' sums apart).
#pragma once

#include "common.cuh"

namespace w4a16 {

constexpr int kTileRows = 16;                    // output rows per MMA tile
constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;  // 256
constexpr int kThreads = kConsumers + 32;        // + one producer warp
constexpr int kChunkGroups = 32;                 // groups per stage (8 boxes)
constexpr int kBoxGroups = 4;                    // 128 bytes of codes per row
constexpr int kBoxBytes = kTileRows * 128;       // 2 KB per TMA box
constexpr int kMaxStages = 16;
constexpr int kMaxSmem = 227 * 1024;
constexpr int kMaxCandidates = 16384;            // pass-2 keys per activation row
constexpr uint32_t kNibPair = 0x000F000Fu;
constexpr uint32_t kNibPairHi = 0x00F000F0u;
constexpr float kTwo24 = 16777216.0f;

__host__ __device__ inline int pow2_at_least(int v) {
    int p = 1;
    while (p < v) p <<= 1;
    return p;
}

__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) & ~(a - 1); }

// ---------------------------------------------------------------------------
// Activation staging.  For local group gl, fragment half h (MMAs j = 2h and
// 2h+1), activation row c and lane quad t, four words are stored at
//   xf[(((gl*2 + h)*M + c)*4 + t)*4 ...]  =  {b0(2h), b1(2h), b0(2h+1), b1(2h+1)}
// with b0(j) = (x[c][k+j], x[c][k+j+4]), b1(j) = (x[c][k+8+j], x[c][k+12+j]),
// k = 64G + 16t.  xsum[gl*M + c] = sum of the group's 64 activations (fp32).
// G32 (group-32 weights): quad t holds instead x[c][64G + 8t .. 8t+7] (half
// 0) and x[c][64G + 32 + 8t ..] (half 1), each as {(x0, x4), (x2, x6),
// (x1, x5) / 16, (x3, x7) / 16} in the same slots (h = half), and
// xsum[(gl*M + c)*2 + h] = the sum of half h.
// The operands of the MMAs for j = 1 and 3 are stored divided by 16 (exact
// for |x| >= 2^-10; below that the halving error is at most 2^-25), because
// their codes are extracted 4 bits higher (see group_mma).
// Run by `nthreads` threads (a multiple of 32) with thread index `tid`.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t sixteenth(uint32_t h2) {
    const __half2 v = __hmul2(*reinterpret_cast<const __half2 *>(&h2), __float2half2_rn(0.0625f));
    return *reinterpret_cast<const uint32_t *>(&v);
}

// 16 tagged activation words (binary16 value in the low half, tag in the
// high half) of one staging item, loaded with relaxed gpu-scope loads until
// every tag equals `tag`.  Bounded: gives up (recording the expiry and
// raising *abort) after the wait limit, or at once when *abort is raised.
// H2: distance in words from the first 8 words to the second 8 (8: one run
// of 16).
template <int H2 = 8>
__device__ __forceinline__ void load_tagged16(const uint32_t *src, uint32_t tag, uint32_t (&v)[16],
                                              volatile int *abort) {
    uint64_t t_start = 0;
    for (uint32_t spin = 0;; ++spin) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
            asm volatile("ld.relaxed.gpu.global.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(v[4 * i]), "=r"(v[4 * i + 1]), "=r"(v[4 * i + 2]), "=r"(v[4 * i + 3])
                         : "l"(src + (i < 2 ? 4 * i : H2 + 4 * (i - 2)))
                         : "memory");
        bool ok = true;
#pragma unroll
        for (int i = 0; i < 16; ++i) ok &= (v[i] >> 16) == tag;
        if (ok) return;
        if (*abort) return;
        if ((spin & 7) == 7) {
            const uint64_t now = global_ns();
            if (t_start == 0) {
                t_start = now;
            } else if (now - t_start > kWaitNs) {
                atomicExch(&g_wait_expired, 1);
                *abort = 1;
                return;
            }
        }
    }
}

// One staging item: 16 activations of row c (two uint4 of half pairs):
// elements e0 .. e0+15, or for G32 e0 .. e0+7 and e0+32 .. e0+39, as read by
// stage_activations_t.
template <bool TAGGED, bool G32 = false>
__device__ __forceinline__ void item_load(const uint16_t *__restrict__ x, const uint32_t *xt, uint32_t tag,
                                          size_t e0, bool coherent, volatile int *abort, uint4 &lo, uint4 &hi) {
    if (TAGGED) {
        uint32_t v[16];
        load_tagged16<G32 ? 32 : 8>(xt + e0, tag, v, abort);
        lo.x = __byte_perm(v[0], v[1], 0x5410);
        lo.y = __byte_perm(v[2], v[3], 0x5410);
        lo.z = __byte_perm(v[4], v[5], 0x5410);
        lo.w = __byte_perm(v[6], v[7], 0x5410);
        hi.x = __byte_perm(v[8], v[9], 0x5410);
        hi.y = __byte_perm(v[10], v[11], 0x5410);
        hi.z = __byte_perm(v[12], v[13], 0x5410);
        hi.w = __byte_perm(v[14], v[15], 0x5410);
    } else {
        const uint4 *src = reinterpret_cast<const uint4 *>(x + e0);
        const uint4 *src2 = G32 ? reinterpret_cast<const uint4 *>(x + e0 + 32) : src + 1;
        lo = coherent ? __ldcg(src) : __ldg(src);
        hi = coherent ? __ldcg(src2) : __ldg(src2);
    }
}

// G32 item: half 0 (lo) and half 1 (hi) in fragment order; returns the sum
// of each half's 8 activations.
__device__ __forceinline__ void item_store_g32(uint4 lo, uint4 hi, int gl, int c, int t, int M, uint32_t *xf,
                                               float &part0, float &part1) {
    auto frag = [](uint4 v) {
        uint4 f;
        f.x = __byte_perm(v.x, v.z, 0x5410);             // (x0, x4)
        f.y = __byte_perm(v.y, v.w, 0x5410);             // (x2, x6)
        f.z = sixteenth(__byte_perm(v.x, v.z, 0x7632));  // (x1, x5) / 16
        f.w = sixteenth(__byte_perm(v.y, v.w, 0x7632));  // (x3, x7) / 16
        return f;
    };
    reinterpret_cast<uint4 *>(xf)[((gl * 2 + 0) * M + c) * 4 + t] = frag(lo);
    reinterpret_cast<uint4 *>(xf)[((gl * 2 + 1) * M + c) * 4 + t] = frag(hi);
    const uint32_t a[4] = {lo.x, lo.y, lo.z, lo.w}, b[4] = {hi.x, hi.y, hi.z, hi.w};
    part0 = part1 = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        part0 += h2f((uint16_t)(a[i] & 0xFFFFu));
        part0 += h2f((uint16_t)(a[i] >> 16));
        part1 += h2f((uint16_t)(b[i] & 0xFFFFu));
        part1 += h2f((uint16_t)(b[i] >> 16));
    }
}

// Stores one item in fragment order; returns the sum of its 16 activations.
__device__ __forceinline__ float item_store(uint4 lo, uint4 hi, int gl, int c, int t, int M, uint32_t *xf) {
    uint4 f0, f1;
    f0.x = __byte_perm(lo.x, lo.z, 0x5410);             // (x0, x4)
    f0.y = __byte_perm(hi.x, hi.z, 0x5410);             // (x8, x12)
    f0.z = sixteenth(__byte_perm(lo.x, lo.z, 0x7632));  // (x1, x5) / 16
    f0.w = sixteenth(__byte_perm(hi.x, hi.z, 0x7632));  // (x9, x13) / 16
    f1.x = __byte_perm(lo.y, lo.w, 0x5410);             // (x2, x6)
    f1.y = __byte_perm(hi.y, hi.w, 0x5410);             // (x10, x14)
    f1.z = sixteenth(__byte_perm(lo.y, lo.w, 0x7632));  // (x3, x7) / 16
    f1.w = sixteenth(__byte_perm(hi.y, hi.w, 0x7632));  // (x11, x15) / 16
    reinterpret_cast<uint4 *>(xf)[((gl * 2 + 0) * M + c) * 4 + t] = f0;
    reinterpret_cast<uint4 *>(xf)[((gl * 2 + 1) * M + c) * 4 + t] = f1;
    const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    float part = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        part += h2f((uint16_t)(w[i] & 0xFFFFu));
        part += h2f((uint16_t)(w[i] >> 16));
    }
    return part;
}

// Activation staging (see the layout above).  TAGGED: read the tagged copy
// `xt` of the activations written earlier in the same launch, waiting for
// the words of tag `tag`; else read x (coherent: bypassing the non-coherent
// read-only path, for activations written earlier in the same kernel).
// A thread takes kB items (it, it + nthreads, ...) together, so their loads
// are in flight at once.
template <bool TAGGED, int kB = 2, bool G32 = false>
__device__ void stage_activations_t(const uint16_t *__restrict__ x, const uint32_t *xt, uint32_t tag, int M, int K,
                                    int g0, int ngl, uint32_t *xf, float *xsum, int tid, int nthreads, bool coherent,
                                    volatile int *abort) {
    const int items = ngl * M * 4;
    for (int base = 0; base < items; base += kB * nthreads) {
        uint4 lo[kB], hi[kB];
#pragma unroll
        for (int u = 0; u < kB; ++u) {
            const int it = base + u * nthreads + tid;
            if (it < items) {
                const int t = it & 3, c = (it >> 2) % M, gl = (it >> 2) / M;
                item_load<TAGGED, G32>(x, xt, tag, (size_t)c * K + (size_t)(g0 + gl) * kGroup + (G32 ? 8 : 16) * t,
                                       coherent, abort, lo[u], hi[u]);
            }
        }
#pragma unroll
        for (int u = 0; u < kB; ++u) {
            const int it = base + u * nthreads + tid;
            if (G32) {
                float p0 = 0.f, p1 = 0.f;
                if (it < items) item_store_g32(lo[u], hi[u], (it >> 2) / M, (it >> 2) % M, it & 3, M, xf, p0, p1);
                p0 += __shfl_xor_sync(0xffffffffu, p0, 1);
                p1 += __shfl_xor_sync(0xffffffffu, p1, 1);
                p0 += __shfl_xor_sync(0xffffffffu, p0, 2);
                p1 += __shfl_xor_sync(0xffffffffu, p1, 2);
                if (it < items && (it & 3) == 0) {
                    xsum[(it >> 2) * 2] = p0;
                    xsum[(it >> 2) * 2 + 1] = p1;
                }
            } else {
                float part = 0.f;
                if (it < items) part = item_store(lo[u], hi[u], (it >> 2) / M, (it >> 2) % M, it & 3, M, xf);
                part += __shfl_xor_sync(0xffffffffu, part, 1);
                part += __shfl_xor_sync(0xffffffffu, part, 2);
                if (it < items && (it & 3) == 0) xsum[it >> 2] = part;
            }
        }
    }
}

template <int kB = 2, bool G32 = false>
__device__ __forceinline__ void stage_activations(const uint16_t *__restrict__ x, int M, int K, int g0, int ngl,
                                                  uint32_t *xf, float *xsum, int tid, int nthreads,
                                                  bool coherent = false) {
    stage_activations_t<false, kB, G32>(x, nullptr, 0u, M, K, g0, ngl, xf, xsum, tid, nthreads, coherent,
                                        nullptr);
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
    // BF: the factor of the bias sums (1; -8 when they hold scale * sum x of
    // symmetric codes, an exact power-of-two scaling).
    template <int BF = 1>
    __device__ __forceinline__ float value(int nt, int i) const {
        return fmaf(kTwo24, s[nt][i], BF == 1 ? b[nt][i] : (float)BF * b[nt][i]);
    }
};

// acc0 += s0 * d0 and acc1 += s1 * d1 in one packed fp32 instruction (each
// lane rounded once, as two fmaf).
__device__ __forceinline__ void ffma2(float &acc0, float &acc1, float s0, float s1, float d0, float d1) {
    asm("{\n .reg .b64 a, s, d;\n mov.b64 a, {%0, %1};\n mov.b64 s, {%2, %3};\n mov.b64 d, {%4, %5};\n"
        " fma.rn.f32x2 a, s, d, a;\n mov.b64 {%0, %1}, a;\n}"
        : "+f"(acc0), "+f"(acc1)
        : "f"(s0), "f"(s1), "f"(d0), "f"(d1));
}

// One group (64 k) of the warp's 16-row tile: 4 MMAs per activation tile.
// wa/wb: words 2t, 2t+1 of rows g and g+8; s*/b*: their scales and biases;
// xl: the lane's staged activation fragments of this group for activation
// tile 0 (column min(g, M-1): lanes past the last activation row repeat it,
// and the MMA columns they produce are never read); xd1: the distance in
// uint4 words to its fragments of tile 1 (column min(8 + g, M-1));
// xs: the group's activation sums.
// M1: a single activation row (only column 0 of the MMA result is used).
template <int NT, bool M1>
__device__ __forceinline__ void group_mma(Acc<NT> &acc, uint2 wa, uint2 wb, float sa, float sb, float ba,
                                          float bb, const uint4 *xl, int xd1, const float *xs, int M, int lt) {
    // Codes j and j+4 of a word as a half pair: even j from (w >> 2j) & 0x000F000F
    // (q * 2^-24), odd j from (w >> 2(j-1)) & 0x00F000F0 (q * 2^-20, matched by
    // activations stored / 16): one shift per word.
    uint32_t a0[4], a1[4], a2[4], a3[4];
    const uint32_t w8[4] = {wa.x >> 8, wb.x >> 8, wa.y >> 8, wb.y >> 8};
    a0[0] = wa.x & kNibPair;  // row g,   cols 2t,2t+1   <- k = 16t+j, +4
    a1[0] = wb.x & kNibPair;  // row g+8, cols 2t,2t+1
    a2[0] = wa.y & kNibPair;  // row g,   cols 2t+8,2t+9 <- k = 16t+8+j, +4
    a3[0] = wb.y & kNibPair;  // row g+8, cols 2t+8,2t+9
    a0[1] = wa.x & kNibPairHi;
    a1[1] = wb.x & kNibPairHi;
    a2[1] = wa.y & kNibPairHi;
    a3[1] = wb.y & kNibPairHi;
    a0[2] = w8[0] & kNibPair;
    a1[2] = w8[1] & kNibPair;
    a2[2] = w8[2] & kNibPair;
    a3[2] = w8[3] & kNibPair;
    a0[3] = w8[0] & kNibPairHi;
    a1[3] = w8[1] & kNibPairHi;
    a2[3] = w8[2] & kNibPairHi;
    a3[3] = w8[3] & kNibPairHi;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        // Fragment half h of column c sits at (h*M + c)*4 + t.
        const int xo = nt ? xd1 : 0;
        const uint4 f0 = xl[xo];
        const uint4 f1 = xl[xo + (M1 ? 4 : M * 4)];
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        mma_16816(d, a0[0], a1[0], a2[0], a3[0], f0.x, f0.y);
        mma_16816(d, a0[1], a1[1], a2[1], a3[1], f0.z, f0.w);
        mma_16816(d, a0[2], a1[2], a2[2], a3[2], f1.x, f1.y);
        mma_16816(d, a0[3], a1[3], a2[3], a3[3], f1.z, f1.w);
        if (M1) {
            // Column 0 lives in d[0] (row g) and d[2] (row g+8) of lanes t = 0.
            const float X0 = xs[0];
            ffma2(acc.s[nt][0], acc.s[nt][2], sa, sb, d[0], d[2]);
            ffma2(acc.b[nt][0], acc.b[nt][2], ba, bb, X0, X0);
        } else {
            const int c0 = min(nt * 8 + 2 * lt, M - 1), c1 = min(nt * 8 + 2 * lt + 1, M - 1);
            const float X0 = xs[c0], X1 = xs[c1];
            ffma2(acc.s[nt][0], acc.s[nt][2], sa, sb, d[0], d[2]);
            ffma2(acc.s[nt][1], acc.s[nt][3], sa, sb, d[1], d[3]);
            ffma2(acc.b[nt][0], acc.b[nt][2], ba, bb, X0, X0);
            ffma2(acc.b[nt][1], acc.b[nt][3], ba, bb, X1, X1);
        }
    }
}

// Group 32: a 64-k group holds two quantisation groups.  Lane (g, t) holds
// word t (k 8t .. 8t+7, half 0) and word t + 4 (half 1) of rows g and g+8:
// wa0, wa1 and wb0, wb1.  Each word feeds two MMAs of its half: codes (0, 4)
// and (2, 6) -- one shift serves the upper byte -- against the staged
// (x0, x4), (x2, x6), and codes (1, 5), (3, 7) at 16x against (x1, x5) / 16,
// (x3, x7) / 16.  So each half's dot products come out of their own two
// MMAs.  sa[h], sb[h], ba[h], bb[h]: scale and bias of half h for rows g and
// g+8; xs[c*2 + h]: half sums of activation row c.
template <int NT, bool M1>
__device__ __forceinline__ void group_mma_g32(Acc<NT> &acc, uint32_t wa0, uint32_t wa1, uint32_t wb0, uint32_t wb1,
                                              const float (&sa)[2], const float (&sb)[2], const float (&ba)[2],
                                              const float (&bb)[2], const uint4 *xl, int xd1, const float *xs, int M,
                                              int lt) {
    // A operands per half: x = codes (0, 4) / (2, 6), y = codes (1, 5) / (3, 7).
    const uint32_t a8 = wa0 >> 8, b8 = wb0 >> 8, c8 = wa1 >> 8, d8 = wb1 >> 8;
    const uint32_t h0x[4] = {wa0 & kNibPair, wb0 & kNibPair, a8 & kNibPair, b8 & kNibPair};
    const uint32_t h0y[4] = {wa0 & kNibPairHi, wb0 & kNibPairHi, a8 & kNibPairHi, b8 & kNibPairHi};
    const uint32_t h1x[4] = {wa1 & kNibPair, wb1 & kNibPair, c8 & kNibPair, d8 & kNibPair};
    const uint32_t h1y[4] = {wa1 & kNibPairHi, wb1 & kNibPairHi, c8 & kNibPairHi, d8 & kNibPairHi};
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int xo = nt ? xd1 : 0;
        const uint4 f0 = xl[xo];                        // half 0 fragments
        const uint4 f1 = xl[xo + (M1 ? 4 : M * 4)];     // half 1 fragments
        float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
        mma_16816(d0, h0x[0], h0x[1], h0x[2], h0x[3], f0.x, f0.y);
        mma_16816(d0, h0y[0], h0y[1], h0y[2], h0y[3], f0.z, f0.w);
        mma_16816(d1, h1x[0], h1x[1], h1x[2], h1x[3], f1.x, f1.y);
        mma_16816(d1, h1y[0], h1y[1], h1y[2], h1y[3], f1.z, f1.w);
        if (M1) {
            ffma2(acc.s[0][0], acc.s[0][2], sa[0], sb[0], d0[0], d0[2]);
            ffma2(acc.s[0][0], acc.s[0][2], sa[1], sb[1], d1[0], d1[2]);
            ffma2(acc.b[0][0], acc.b[0][2], ba[0], bb[0], xs[0], xs[0]);
            ffma2(acc.b[0][0], acc.b[0][2], ba[1], bb[1], xs[1], xs[1]);
        } else {
            const int c0 = min(nt * 8 + 2 * lt, M - 1), c1 = min(nt * 8 + 2 * lt + 1, M - 1);
            ffma2(acc.s[nt][0], acc.s[nt][2], sa[0], sb[0], d0[0], d0[2]);
            ffma2(acc.s[nt][0], acc.s[nt][2], sa[1], sb[1], d1[0], d1[2]);
            ffma2(acc.s[nt][1], acc.s[nt][3], sa[0], sb[0], d0[1], d0[3]);
            ffma2(acc.s[nt][1], acc.s[nt][3], sa[1], sb[1], d1[1], d1[3]);
            ffma2(acc.b[nt][0], acc.b[nt][2], ba[0], bb[0], xs[2 * c0], xs[2 * c0]);
            ffma2(acc.b[nt][0], acc.b[nt][2], ba[1], bb[1], xs[2 * c0 + 1], xs[2 * c0 + 1]);
            ffma2(acc.b[nt][1], acc.b[nt][3], ba[0], bb[0], xs[2 * c1], xs[2 * c1]);
            ffma2(acc.b[nt][1], acc.b[nt][3], ba[1], bb[1], xs[2 * c1 + 1], xs[2 * c1 + 1]);
        }
    }
}

// Group 32: byte offset, within a stage, of word t of row g in box `box`
// (group j adds ((2j + h) ^ (g % 8)) << 4 for half h; row g+8 is 1024 bytes
// further with the same swizzle phase).
__device__ __forceinline__ int g32_offset(int box, int lg, int lt) { return box * kBoxBytes + lg * 128 + 4 * lt; }

// Shared-memory byte offsets, within a stage, of the words a lane reads for
// group j (0..3) of box `box`: row g, 16-byte chunk 2j + t/2 under the
// 128-byte swizzle (chunk index XOR row % 8), word pair t % 2.  Row g+8 is
// 1024 bytes further with the same swizzle phase.
__device__ __forceinline__ void box_offsets(int (&off)[4], int box, int lg, int lt) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
        off[j] = box * kBoxBytes + lg * 128 + ((((2 * j) | (lt >> 1)) ^ (lg & 7)) << 4) + ((lt & 1) << 3);
}

__device__ __forceinline__ void unpack4h(uint2 v, float (&f)[4]) {
    const float2 lo = __half22float2(*reinterpret_cast<const __half2 *>(&v.x));
    const float2 hi = __half22float2(*reinterpret_cast<const __half2 *>(&v.y));
    f[0] = lo.x;
    f[1] = lo.y;
    f[2] = hi.x;
    f[3] = hi.y;
}

// Whether a full box (4 groups from a multiple of 4) can read its scales as
// one aligned vector: the rows' scale arrays keep that alignment.  (For
// group 64 this is K % 256 == 0.)
__host__ __device__ inline bool box_vec_ok(const WFmt &f) {
    if (f.gs == 0) return f.ngs % 8 == 0;  // 8 scales per row: 16 bytes
    if (f.gs == 1) return f.ngs % 4 == 0;  // 4 scales: 8 bytes
    if (f.gs == 2) return f.ngs % 2 == 0;  // 2 scales: 4 bytes
    return true;                           // one scale
}

// Scale and bias of groups g .. g+3 (entries j < n) of rows g and g+8 (lane
// row lg): one quantisation group spans 1 << (gs - 1) groups (gs >= 1).
// sp: the tile's scales [16][ngs], followed by its biases unless f.sym
// (then bias = -8 * scale, exact in fp32).
template <bool FULL>
__device__ __forceinline__ void box_scales(float (&fsa)[4], float (&fsb)[4], float (&fba)[4], float (&fbb)[4],
                                           const uint16_t *sp, const WFmt &f, int g, int n, int lg) {
    const int ngs = f.ngs, sh = f.gs - 1;
    const uint16_t *ra = sp + lg * ngs;
    const uint16_t *rb = ra + 8 * ngs;
    auto load = [&](const uint16_t *r, float (&o)[4]) {
        if (FULL && sh == 0) {
            unpack4h(*reinterpret_cast<const uint2 *>(r + g), o);
        } else if (FULL && sh == 1) {
            const float2 v = __half22float2(*reinterpret_cast<const __half2 *>(r + (g >> 1)));
            o[0] = o[1] = v.x;
            o[2] = o[3] = v.y;
        } else if (FULL) {
            o[0] = o[1] = o[2] = o[3] = h2f(r[g >> sh]);
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) o[j] = h2f(r[(g + (j < n ? j : 0)) >> sh]);
        }
    };
    load(ra, fsa);
    load(rb, fsb);
    if (f.sym) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            fba[j] = -8.f * fsa[j];
            fbb[j] = -8.f * fsb[j];
        }
    } else {
        load(ra + kTileRows * ngs, fba);
        load(rb + kTileRows * ngs, fbb);
    }
}

// Group 32: the two halves' scales (and biases) of groups g .. g+3.
template <bool FULL>
__device__ __forceinline__ void box_scales_g32(float (&fsa)[4][2], float (&fsb)[4][2], float (&fba)[4][2],
                                               float (&fbb)[4][2], const uint16_t *sp, const WFmt &f, int g, int n,
                                               int lg) {
    const int ngs = f.ngs;
    const uint16_t *ra = sp + lg * ngs;
    const uint16_t *rb = ra + 8 * ngs;
    auto load = [&](const uint16_t *r, float (&o)[4][2]) {
        if (FULL) {
            const uint4 v = *reinterpret_cast<const uint4 *>(r + 2 * g);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float2 p = __half22float2(*reinterpret_cast<const __half2 *>(&w[j]));
                o[j][0] = p.x;
                o[j][1] = p.y;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int jj = j < n ? j : 0;
                o[j][0] = h2f(r[2 * (g + jj)]);
                o[j][1] = h2f(r[2 * (g + jj) + 1]);
            }
        }
    };
    load(ra, fsa);
    load(rb, fsb);
    if (f.sym) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                fba[j][h] = -8.f * fsa[j][h];
                fbb[j][h] = -8.f * fsb[j][h];
            }
    } else {
        load(ra + kTileRows * ngs, fba);
        load(rb + kTileRows * ngs, fbb);
    }
}

// The warp's box of a stage: n (1..4) consecutive groups of a 16-row tile.
// st: the stage; sp: the tile's scales and biases (see box_scales);
// g: the box's first group; xl: the lane's staged activation fragments of
// that group (see group_mma); xs: its activation sums.  FULL: n == 4 and
// box_vec_ok(f).  FMT: kFmtG64 reads one scale and one bias per group
// (f.ngs groups per row), kFmtS128 one scale per two groups and no bias (the
// bias sums then accumulate scale * sum x: see Acc::value), kFmtAny follows
// f, kFmtG32 is the group-32 variant (goff: see g32_offset).
template <int NT, bool M1, bool FULL, int FMT>
__device__ __forceinline__ void box_mma(Acc<NT> &acc, const uint8_t *st, const int (&off)[4], const uint16_t *sp,
                                        const WFmt &f, int g, int n, const uint4 *xl, int xd1, const float *xs,
                                        int M, int lg, int lt, int goff = 0) {
    const int xstep = 2 * M * 4;  // uint4 words of staged activations per group
    if (FMT == kFmtG32) {
        float fsa[4][2], fsb[4][2], fba[4][2], fbb[4][2];
        box_scales_g32<FULL>(fsa, fsb, fba, fbb, sp, f, g, n, lg);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (FULL || j < n) {
                const uint8_t *p0 = st + goff + ((((2 * j) ^ (lg & 7))) << 4);
                const uint8_t *p1 = st + goff + ((((2 * j + 1) ^ (lg & 7))) << 4);
                const uint32_t wa0 = *reinterpret_cast<const uint32_t *>(p0);
                const uint32_t wa1 = *reinterpret_cast<const uint32_t *>(p1);
                const uint32_t wb0 = *reinterpret_cast<const uint32_t *>(p0 + 8 * 128);
                const uint32_t wb1 = *reinterpret_cast<const uint32_t *>(p1 + 8 * 128);
                group_mma_g32<NT, M1>(acc, wa0, wa1, wb0, wb1, fsa[j], fsb[j], fba[j], fbb[j],
                                      xl + j * (M1 ? 8 : xstep), xd1, xs + j * 2 * M, M, lt);
            }
        }
        return;
    }
    float fsa[4], fsb[4], fba[4], fbb[4];
    if (FMT == kFmtG64) {
        const int ng = f.ngs;
        const uint16_t *sa = sp + lg * ng + g;  // scales of row g; row g+8 is 8 rows on
        const uint16_t *ba = sa + kTileRows * ng;
        if (FULL) {
            unpack4h(*reinterpret_cast<const uint2 *>(sa), fsa);
            unpack4h(*reinterpret_cast<const uint2 *>(sa + 8 * ng), fsb);
            unpack4h(*reinterpret_cast<const uint2 *>(ba), fba);
            unpack4h(*reinterpret_cast<const uint2 *>(ba + 8 * ng), fbb);
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int jj = j < n ? j : 0;
                fsa[j] = h2f(sa[jj]);
                fsb[j] = h2f(sa[8 * ng + jj]);
                fba[j] = h2f(ba[jj]);
                fbb[j] = h2f(ba[8 * ng + jj]);
            }
        }
    } else if (FMT == kFmtS128) {
        const int ngs = f.ngs;
        const uint16_t *sa = sp + lg * ngs;
        if (FULL) {
            const float2 va = __half22float2(*reinterpret_cast<const __half2 *>(sa + (g >> 1)));
            const float2 vb = __half22float2(*reinterpret_cast<const __half2 *>(sa + 8 * ngs + (g >> 1)));
            fsa[0] = fsa[1] = va.x;
            fsa[2] = fsa[3] = va.y;
            fsb[0] = fsb[1] = vb.x;
            fsb[2] = fsb[3] = vb.y;
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int gj = (g + (j < n ? j : 0)) >> 1;
                fsa[j] = h2f(sa[gj]);
                fsb[j] = h2f(sa[8 * ngs + gj]);
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            fba[j] = fsa[j];
            fbb[j] = fsb[j];
        }
    } else {
        box_scales<FULL>(fsa, fsb, fba, fbb, sp, f, g, n, lg);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        if (FULL || j < n) {
            const uint2 wa = *reinterpret_cast<const uint2 *>(st + off[j]);
            const uint2 wb = *reinterpret_cast<const uint2 *>(st + off[j] + 8 * 128);
            group_mma<NT, M1>(acc, wa, wb, fsa[j], fsb[j], fba[j], fbb[j], xl + j * (M1 ? 8 : xstep), xd1,
                              xs + j * (M1 ? 1 : M), M, lt);
        }
    }
}

// Offset (uint4 words) of the lane's activation fragments within a group's
// block: column min(g, M-1) of tile 0, quad t.
__device__ __forceinline__ int lane_xoff(int M, int lg, int lt) { return min(lg, M - 1) * 4 + lt; }
// Distance from those to the lane's fragments of tile 1 (column min(8+g, M-1)).
__device__ __forceinline__ int lane_xd1(int M, int lg) { return (min(8 + lg, M - 1) - min(lg, M - 1)) * 4; }

}  // namespace w4a16
