// Packed variable-length QK rotary position embedding for GB300 (sm_103a).
//
// One CTA owns a tile of consecutive tokens and rotates every Q head and every K head
// of those tokens (grouped-query attention: any n_q_heads / n_kv_heads).  Per tile:
//   1. the first warp finds each token's sample by binary search over cu_seqlens, so
//      positions restart at every packed-sample boundary (unsloth.ai "3x faster
//      training with packing", section "Packing non contaminé");
//   2. the (cos, sin) rows of the tile's positions are staged once in shared memory,
//      from the caller's cache or evaluated on the fly (both give the same bits), and
//      shared by all heads;
//   3. all threads stream Q then K rows with 16-byte loads and stores: each thread
//      takes 8 elements from each half of a head and applies
//        y = x*cos + rotate_half(x)*sin    (section "Kernel Triton QK RoPE fusionné
//      avec packing"), the backward being the same with sin negated (R^T).
// The work is HBM-bound (about 0.75 flop per byte), so there are no tensor cores and
// no fusion into a contraction.  64-bit flat offsets are a compile-time
// specialisation, used only when an element count reaches 2^31 (section "Indexage
// int64 pour les kernels Triton").
//
// Every floating-point step is an explicit round-to-nearest intrinsic so that the
// compiler cannot contract a multiply and an add; results are bit-identical to a plain
// sequential evaluation of the same steps on a CPU.
//
// Launches use programmatic dependent launch: a grid may be scheduled while the
// previous kernel in its stream drains, and its first instruction waits for that
// kernel to complete, so back-to-back rotations lose no launch gap and nothing is read
// early.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <type_traits>
#include <utility>

#include "cos_sin.cuh"
#include "fastdiv.cuh"
#include "rope_qk.h"

namespace {

constexpr int kThreads = 128;           // threads per CTA (9 CTAs per SM at 56 registers)
constexpr int kTileUnits = 512;         // about this many 16-byte pair units per tile
constexpr int kWideGrid = 32768;        // tiles from which a launch with a cos/sin cache
                                        // keeps 4 pair units in flight per thread (below:
                                        // 3 or 2), and keeps full-size tiles
constexpr int kMaxHalf = 128;           // head_dim <= 256
constexpr int kMaxTileTokens = 32;      // one warp resolves the tile's positions
constexpr int kMaxSegments = ROPE_MAX_SEGMENTS;
constexpr int kMaxStagedCu = 256;       // cu_seqlens entries a CTA copies to shared memory
constexpr int64_t kMaxTokens = int64_t(1) << 24;   // positions < 2^24 are exact in fp32

using pvr::FastDiv;
using pvr::fast_div;
using pvr::make_fastdiv;

struct RopeArgs {
    const __nv_bfloat16 *q_in;
    const __nv_bfloat16 *k_in;
    __nv_bfloat16 *q_out;
    __nv_bfloat16 *k_out;
    int64_t q_ts, q_hs, k_ts, k_hs;          // input strides in elements (token, head)
    int64_t qo_ts, qo_hs, ko_ts, ko_hs;      // output strides
    const int32_t *cu;
    const int32_t *pos_ids;                  // optional per-row positions (replaces cu)
    const long long *pos_ids64;              // the same as int64 values
    const int32_t *seq_used;                 // optional tokens used per sample (with cu)
    const float4 *cache;
    int32_t n_seqs;
    int32_t stage_cu;                        // cu_seqlens staged in shared memory (n_seqs < kMaxStagedCu)
    int32_t n_tokens;
    int32_t n_seg;                           // >= 1 row segments (cu_seqlens positions)
    int32_t seg_row[kMaxSegments];           // first row of segment i (seg_row[0] == 0)
    int32_t seg_delta[kMaxSegments];         // row r of segment i is token r + seg_delta[i]
    int32_t hq;
    int32_t hkv;
    int32_t h_tot;
    int32_t head_dim;
    int32_t cache_rows;
    int32_t tile_tokens;
    int32_t in_place;
    int32_t bwd;
    FastDiv div_htot;
    FastDiv div_cph;
    float w[kMaxHalf];
};

// Position of token t: t - cu[s] for the last s in [0, n) with cu[s] <= t, or -1 when
// t lies outside [cu[0], cu[n]) or, given seq_used, at or past seq_used[s] tokens into
// its sample.  The loop is bounded by log2(n) steps whatever cu holds; a result that
// would not be a valid position (start < 0 or start > t, only possible for a cu that is
// not non-decreasing) is reported as outside.
__device__ __forceinline__ int token_position(const int32_t *__restrict__ cu, int n, int t,
                                              const int32_t *__restrict__ seq_used = nullptr)
{
    if (n <= 0) return -1;
    const int first = __ldg(cu);
    const int last = __ldg(cu + n);
    if (t < first || t >= last) return -1;
    int lo = 0, hi = n;
    while (hi - lo > 1) {
        const int mid = lo + ((hi - lo) >> 1);
        if (__ldg(cu + mid) <= t) lo = mid;
        else hi = mid;
    }
    const int start = __ldg(cu + lo);
    if (start < 0 || start > t) return -1;
    const int pos = t - start;
    if (seq_used != nullptr && pos >= __ldg(seq_used + lo)) return -1;
    return pos;
}

// token_position over a copy of cu_seqlens in shared memory (same rules).
__device__ __forceinline__ int token_position_staged(const int32_t *cu, int n, int t,
                                                     const int32_t *__restrict__ seq_used)
{
    if (n <= 0) return -1;
    if (t < cu[0] || t >= cu[n]) return -1;
    int lo = 0, hi = n;
    while (hi - lo > 1) {
        const int mid = lo + ((hi - lo) >> 1);
        if (cu[mid] <= t) lo = mid;
        else hi = mid;
    }
    const int start = cu[lo];
    if (start < 0 || start > t) return -1;
    const int pos = t - start;
    if (seq_used != nullptr && pos >= __ldg(seq_used + lo)) return -1;
    return pos;
}

// (cos phi, sin phi) of a binary32 angle in binary64, each rounded once to binary32.
__device__ __noinline__ float2 cos_sin_binary64(float phi)
{
    double s, c;
    sincos(static_cast<double>(phi), &s, &c);
    return make_float2(__double2float_rn(c), __double2float_rn(s));
}

// (cos phi, sin phi) with phi = RN32(pos * w): the angle is one binary32 multiply; the
// cosine and sine are the binary64 values rounded once to binary32, obtained in
// binary32 double-float arithmetic where its rounding is certain (all but a few cases
// in a million) and in binary64 otherwise.
__device__ __forceinline__ float2 cos_sin_of(float phi)
{
    float c, s;
    if (pvr::cos_sin_binary32(phi, c, s)) return make_float2(c, s);
    return cos_sin_binary64(phi);
}

__device__ __forceinline__ float2 cos_sin_at(int pos, float w)
{
    return cos_sin_of(__fmul_rn(__int2float_rn(pos), w));
}

__device__ __forceinline__ uint4 load_stream(const __nv_bfloat16 *p)
{
    return __ldcs(reinterpret_cast<const uint4 *>(p));
}

__device__ __forceinline__ void store_stream(__nv_bfloat16 *p, uint4 v)
{
    __stcs(reinterpret_cast<uint4 *>(p), v);
}

__device__ __forceinline__ uint32_t bf162_bits(__nv_bfloat162 v)
{
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ __nv_bfloat162 bits_bf162(uint32_t u)
{
    return *reinterpret_cast<__nv_bfloat162 *>(&u);
}

// Rotate two bf16 pairs: a = first-half elements, b = second-half elements, with
// (c0, s0, c1, s1) for the two frequencies.  lo' = a*c - b*s, hi' = b*c + a*s.
__device__ __forceinline__ void rotate2(uint32_t &lo, uint32_t &hi, float4 cs)
{
    const __nv_bfloat162 a = bits_bf162(lo);
    const __nv_bfloat162 b = bits_bf162(hi);
    const float a0 = __low2float(a), a1 = __high2float(a);
    const float b0 = __low2float(b), b1 = __high2float(b);
    const float y0 = __fsub_rn(__fmul_rn(a0, cs.x), __fmul_rn(b0, cs.y));
    const float z0 = __fadd_rn(__fmul_rn(b0, cs.x), __fmul_rn(a0, cs.y));
    const float y1 = __fsub_rn(__fmul_rn(a1, cs.z), __fmul_rn(b1, cs.w));
    const float z1 = __fadd_rn(__fmul_rn(b1, cs.z), __fmul_rn(a1, cs.w));
    lo = bf162_bits(__floats2bfloat162_rn(y0, y1));
    hi = bf162_bits(__floats2bfloat162_rn(z0, z1));
}

// Shared-memory (cos, sin) rows of a tile use the cache's layout: per token, float4
// entries [quad][chunk] where chunk c covers frequencies 8c..8c+7 and quad q holds
// (cos, sin) of frequencies 8c+2q and 8c+2q+1.  The eight threads of a 16-byte load
// phase (consecutive chunks of one head) read eight consecutive float4: no bank
// conflicts.
template <int D, bool LONG, int U>
__global__ void __launch_bounds__(kThreads)
rope_qk_tile_kernel(const __grid_constant__ RopeArgs a)
{
    using Index = typename std::conditional<LONG, int64_t, uint32_t>::type;
    extern __shared__ __align__(16) float4 s_cs[];
    __shared__ int s_pos[kMaxTileTokens];

    const int d = D > 0 ? D : a.head_dim;
    const int h = d >> 1;
    const int cph = d >> 4;
    const int row4 = 4 * cph;
    const int t0 = blockIdx.x * a.tile_tokens;
    const int tt = min(a.tile_tokens, a.n_tokens - t0);
    const uint32_t units = static_cast<uint32_t>(tt) * static_cast<uint32_t>(a.h_tot * cph);

    // A unit is 8 elements from each half of one head of one token: (token i, virtual
    // head vh in [0, hq + hkv), chunk c).  Its input and output addresses:
    auto locate = [&](uint32_t u, uint32_t &i, uint32_t &c, const __nv_bfloat16 *&src, __nv_bfloat16 *&dst) {
        const uint32_t hr = D > 0 ? u / static_cast<uint32_t>(D >> 4) : fast_div(u, a.div_cph);
        c = u - hr * static_cast<uint32_t>(cph);
        i = fast_div(hr, a.div_htot);
        const uint32_t vh = hr - i * static_cast<uint32_t>(a.h_tot);
        const Index t = static_cast<Index>(t0) + static_cast<Index>(i);
        const Index e = static_cast<Index>(c * 8);
        if (vh < static_cast<uint32_t>(a.hq)) {
            const Index hd = static_cast<Index>(vh);
            src = a.q_in + (t * static_cast<Index>(a.q_ts) + hd * static_cast<Index>(a.q_hs) + e);
            dst = a.q_out + (t * static_cast<Index>(a.qo_ts) + hd * static_cast<Index>(a.qo_hs) + e);
        } else {
            const Index hd = static_cast<Index>(vh - a.hq);
            src = a.k_in + (t * static_cast<Index>(a.k_ts) + hd * static_cast<Index>(a.k_hs) + e);
            dst = a.k_out + (t * static_cast<Index>(a.ko_ts) + hd * static_cast<Index>(a.ko_hs) + e);
        }
    };

    // Programmatic dependent launch: the grid may be scheduled while the kernel before
    // it in the stream drains; nothing is read before that kernel has completed and its
    // writes are visible, and the next launch may be scheduled from here on (a no-op
    // for a plain launch).
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    // 0. the tile's first batch of Q/K units (U per thread) is loaded before the
    //    positions are known: the loads do not depend on them, so HBM starts streaming
    //    while the position search and the cos/sin staging run.  An in-place row found
    //    to lie outside the pack is then simply not stored.  With seq_used (a padded
    //    batch whose pad rows are left out), whole tiles may hold no row to rotate, so
    //    the first batch waits for the positions there and skips those rows' loads.
    const bool early = a.seq_used == nullptr;
    uint4 first_lo[U], first_hi[U];
    __nv_bfloat16 *first_dst[U];
    uint32_t first_tok[U], first_chunk[U];
#pragma unroll
    for (int k = 0; k < U; ++k) {
        const uint32_t u = threadIdx.x + k * kThreads;
        first_dst[k] = nullptr;
        first_tok[k] = 0;
        first_chunk[k] = 0;
        if (early && u < units) {
            const __nv_bfloat16 *src;
            locate(u, first_tok[k], first_chunk[k], src, first_dst[k]);
            first_lo[k] = load_stream(src);
            first_hi[k] = load_stream(src + h);
        }
    }

    // 1. positions of the tile's tokens (one lane per token): from the caller's
    //    position ids, else by binary search of cu_seqlens in the global token stream --
    //    in a copy the CTA makes in shared memory with one coalesced round of loads when
    //    it is short, so that the search costs one global round trip instead of log2(n)
    //    dependent ones
    int32_t *s_cu = reinterpret_cast<int32_t *>(s_cs + a.tile_tokens * row4);
    if (a.stage_cu) {
        for (int i = threadIdx.x; i <= a.n_seqs; i += kThreads) s_cu[i] = __ldg(a.cu + i);
        __syncthreads();
    }
    int lane_pos = -1;
    if (threadIdx.x < kMaxTileTokens) {
        int pos = -1;
        if (static_cast<int>(threadIdx.x) < tt) {
            const int r = t0 + static_cast<int>(threadIdx.x);
            if (a.pos_ids != nullptr) {
                const int p = __ldg(a.pos_ids + r);
                pos = (p >= 0 && p < static_cast<int>(kMaxTokens)) ? p : -1;
            } else if (a.pos_ids64 != nullptr) {
                const long long p = __ldg(a.pos_ids64 + r);
                pos = (p >= 0 && p < static_cast<long long>(kMaxTokens)) ? static_cast<int>(p) : -1;
            } else {
                int seg = 0;
                for (int i = 1; i < a.n_seg; ++i)
                    if (r >= a.seg_row[i]) seg = i;
                pos = a.stage_cu ? token_position_staged(s_cu, a.n_seqs, r + a.seg_delta[seg], a.seq_used)
                                 : token_position(a.cu, a.n_seqs, r + a.seg_delta[seg], a.seq_used);
            }
        }
        s_pos[threadIdx.x] = pos;
        lane_pos = pos;
    }
    // A tile with no token inside the pack (the pad rows of a padded batch under
    // seq_used, rows past the pack's end) has nothing to rotate: in place, it is done.
    if (!__syncthreads_or(lane_pos >= 0) && a.in_place) return;

    // 2. (cos, sin) rows of the tile, sin negated for the backward.  A row is 4*cph
    //    float4 in the cache's own [quad][chunk] order, so staging is a plain copy; when
    //    evaluated, each thread takes one (cos, sin) pair (half of a float4 entry), so
    //    twice as many threads share the evaluation.
    if (a.cache != nullptr) {
        for (int idx = threadIdx.x; idx < tt * row4; idx += kThreads) {
            const int i = idx / row4;
            const int r = idx - i * row4;
            const int pos = s_pos[i];
            float4 cs = make_float4(1.0f, 0.0f, 1.0f, 0.0f);
            if (pos >= 0) {
                if (pos < a.cache_rows) {
                    cs = __ldg(a.cache + static_cast<int64_t>(pos) * row4 + r);
                } else {
                    const int quad = r / cph;
                    const int j = 8 * (r - quad * cph) + 2 * quad;
                    const float2 c0 = cos_sin_at(pos, a.w[j]);
                    const float2 c1 = cos_sin_at(pos, a.w[j + 1]);
                    cs = make_float4(c0.x, c0.y, c1.x, c1.y);
                }
                if (a.bwd) {
                    cs.y = -cs.y;
                    cs.w = -cs.w;
                }
            }
            s_cs[idx] = cs;
        }
    } else {
        float2 *s_cs2 = reinterpret_cast<float2 *>(s_cs);
        for (int p2 = threadIdx.x; p2 < 2 * tt * row4; p2 += kThreads) {
            const int idx = p2 >> 1;
            const int i = idx / row4;
            const int r = idx - i * row4;
            const int pos = s_pos[i];
            float2 cs = make_float2(1.0f, 0.0f);
            if (pos >= 0) {
                const int quad = r / cph;
                const int j = 8 * (r - quad * cph) + 2 * quad + (p2 & 1);
                cs = cos_sin_at(pos, a.w[j]);
                if (a.bwd) cs.y = -cs.y;
            }
            s_cs2[p2] = cs;
        }
    }
    __syncthreads();

    // 3. stream the tile: rotate and store the first batch, then load a batch of units
    //    (U per thread, 4 loads of 16 B in flight), rotate, store, and so on.  Rows
    //    of tokens outside the pack are not touched in place and are copied unchanged
    //    out of place.
    if (!early) {
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const uint32_t u = threadIdx.x + k * kThreads;
            if (u >= units) continue;
            const __nv_bfloat16 *src;
            __nv_bfloat16 *out;
            locate(u, first_tok[k], first_chunk[k], src, out);
            if (s_pos[first_tok[k]] < 0 && a.in_place) continue;
            first_dst[k] = out;
            first_lo[k] = load_stream(src);
            first_hi[k] = load_stream(src + h);
        }
    }
#pragma unroll
    for (int k = 0; k < U; ++k) {
        if (first_dst[k] == nullptr) continue;
        const int pos = s_pos[first_tok[k]];
        if (pos < 0 && a.in_place) continue;
        if (pos >= 0) {
            const float4 *cs = s_cs + (static_cast<int>(first_tok[k]) * 4) * cph + first_chunk[k];
            rotate2(first_lo[k].x, first_hi[k].x, cs[0]);
            rotate2(first_lo[k].y, first_hi[k].y, cs[cph]);
            rotate2(first_lo[k].z, first_hi[k].z, cs[2 * cph]);
            rotate2(first_lo[k].w, first_hi[k].w, cs[3 * cph]);
        }
        store_stream(first_dst[k], first_lo[k]);
        store_stream(first_dst[k] + h, first_hi[k]);
    }
    for (uint32_t base = threadIdx.x + U * kThreads; base < units; base += U * kThreads) {
        uint4 lo[U], hi[U];
        __nv_bfloat16 *dst[U];
        int tok[U], chunk[U];
        bool live[U];
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const uint32_t u = base + k * kThreads;
            live[k] = false;
            tok[k] = -1;
            chunk[k] = 0;
            dst[k] = nullptr;
            if (u < units) {
                uint32_t i, c;
                const __nv_bfloat16 *src;
                __nv_bfloat16 *out;
                locate(u, i, c, src, out);
                const int pos = s_pos[i];
                if (pos >= 0 || !a.in_place) {
                    lo[k] = load_stream(src);
                    hi[k] = load_stream(src + h);
                    live[k] = true;
                    dst[k] = out;
                    tok[k] = pos >= 0 ? static_cast<int>(i) : -1;
                    chunk[k] = static_cast<int>(c);
                }
            }
        }
#pragma unroll
        for (int k = 0; k < U; ++k) {
            if (!live[k]) continue;
            if (tok[k] >= 0) {
                const float4 *cs = s_cs + (tok[k] * 4) * cph + chunk[k];
                rotate2(lo[k].x, hi[k].x, cs[0]);
                rotate2(lo[k].y, hi[k].y, cs[cph]);
                rotate2(lo[k].z, hi[k].z, cs[2 * cph]);
                rotate2(lo[k].w, hi[k].w, cs[3 * cph]);
            }
            store_stream(dst[k], lo[k]);
            store_stream(dst[k] + h, hi[k]);
        }
    }
}

struct CacheArgs {
    float w[kMaxHalf];
};

// One float4 entry (cos, sin of frequencies j and j+1, j = 8*chunk + 2*quad) per
// thread, in the [row][quad][chunk] order the rotation kernel stages.
__global__ void cos_sin_cache_kernel(float4 *__restrict__ cache, int64_t rows, int cph,
                                     const __grid_constant__ CacheArgs a)
{
    const int row4 = 4 * cph;
    const int64_t n = rows * row4;
    for (int64_t idx = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; idx < n;
         idx += int64_t(gridDim.x) * blockDim.x) {
        const int64_t p = idx / row4;
        const int r = static_cast<int>(idx - p * row4);
        const int quad = r / cph;
        const int j = 8 * (r - quad * cph) + 2 * quad;
        const float2 c0 = cos_sin_at(static_cast<int>(p), a.w[j]);
        const float2 c1 = cos_sin_at(static_cast<int>(p), a.w[j + 1]);
        cache[idx] = make_float4(c0.x, c0.y, c1.x, c1.y);
    }
}

__global__ void positions_kernel(const int32_t *__restrict__ cu, int n, int n_tokens,
                                 int32_t *__restrict__ pos_out)
{
    for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < n_tokens; t += gridDim.x * blockDim.x)
        pos_out[t] = token_position(cu, n, t);
}

__global__ void validate_kernel(const int32_t *__restrict__ cu, int n, int64_t n_tokens,
                                int32_t *__restrict__ err)
{
    int32_t bits = 0;
    const int64_t tid = blockIdx.x * int64_t(blockDim.x) + threadIdx.x;
    for (int64_t s = tid; s < n; s += int64_t(gridDim.x) * blockDim.x)
        if (__ldg(cu + s + 1) < __ldg(cu + s)) bits |= ROPE_CU_DECREASING;
    if (tid == 0) {
        const int first = __ldg(cu);
        if (first < 0) bits |= ROPE_CU_NEGATIVE_START;
        if (first != 0) bits |= ROPE_CU_NONZERO_START;
        if (static_cast<int64_t>(__ldg(cu + n)) > n_tokens) bits |= ROPE_CU_PAST_END;
    }
    if (bits) atomicOr(err, bits);
}

// cos/sin of given angles: mode 0 as the rotation evaluates them, 1 in binary64 only,
// 2 in binary32 only (NaN where that defers to binary64).
__global__ void cos_sin_eval_kernel(const float *__restrict__ phi, float *__restrict__ c_out,
                                    float *__restrict__ s_out, int64_t n, int mode)
{
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n; i += int64_t(gridDim.x) * blockDim.x) {
        const float x = phi[i];
        float2 cs;
        if (mode == 0) {
            cs = cos_sin_of(x);
        } else if (mode == 1) {
            cs = cos_sin_binary64(x);
        } else {
            float c, s;
            cs = pvr::cos_sin_binary32(x, c, s) ? make_float2(c, s) : make_float2(__int_as_float(0x7fc00000),
                                                                                  __int_as_float(0x7fc00000));
        }
        c_out[i] = cs.x;
        s_out[i] = cs.y;
    }
}

// ------------------------------------------------------------------ host side

// w_j = RN32( pow(theta, -(2j)/d) / scale ), binary64 until the one rounding; a linear
// position rescale by `scale` (position p acts as p / scale) divides every frequency.
void host_inv_freq(double theta, int d, double scale, float *w)
{
    for (int j = 0; j < d / 2; ++j)
        w[j] = static_cast<float>(std::pow(theta, -(2.0 * static_cast<double>(j)) / static_cast<double>(d)) / scale);
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool overlap(const void *a, int64_t na, const void *b, int64_t nb)
{
    if (na <= 0 || nb <= 0) return false;
    const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
    return pa < pb + static_cast<uintptr_t>(nb) && pb < pa + static_cast<uintptr_t>(na);
}

int check_head_dim(int32_t head_dim)
{
    if (head_dim < 16 || head_dim > 2 * kMaxHalf || head_dim % 16 != 0) return ROPE_ERR_HEAD_DIM;
    return ROPE_OK;
}

int check_theta(double theta)
{
    if (!(theta > 0.0) || !std::isfinite(theta)) return ROPE_ERR_THETA;
    return ROPE_OK;
}

int check_scale(double scale)
{
    if (!(scale > 0.0) || !std::isfinite(scale)) return ROPE_ERR_THETA;
    return ROPE_OK;
}

// Pair units per tile for a launch of fewer than kWideGrid such tiles whose cos/sin rows
// are read from a cache and whose rows all have work (no seq_used): half of kTileUnits.
constexpr int kTileUnitsCached = kTileUnits / 2;
// Pair units per tile under seq_used (a padded batch whose pad rows are skipped): twice
// kTileUnits, so that fewer CTAs are spent on tiles of pad rows only (4-token tiles on
// 40 heads of 128: 29.03 -> 28.58 us on 8 x 2048 rows, 47 % valid; 7-token tiles 29.0).
constexpr int kTileUnitsSeqUsed = 2 * kTileUnits;

// Tokens per tile: about `target` 16-byte pair units, capped by the one-warp position
// search.  The targets: kTileUnits (two batches of 2 units per thread) by default,
// twice that under seq_used, half of it for short cached launches.  Half gives 1-token
// tiles on 40 heads of 128 and a shorter drain at the launch's end: 1.5 % faster on
// 16,384 tokens and 1-2 % on a context-parallel rank's half of it with a cos/sin cache,
// but 2.6 % slower without one, 20 % slower on a padded batch under seq_used (there
// each tile's position search and cos/sin staging serve half as many tokens), and
// 6-16 % slower on launches of 100,000+ tokens with head_dim 64, 80 or 128, where the
// per-tile prologue outweighs the drain.
int pick_tile_tokens(int h_tot, int head_dim, int target)
{
    const int units_per_token = h_tot * (head_dim / 16);
    int tt = (target + units_per_token - 1) / units_per_token;
    if (tt < 1) tt = 1;
    if (tt > kMaxTileTokens) tt = kMaxTileTokens;
    return tt;
}

// With `pdl`, the launch carries the programmatic-stream-serialisation attribute:
// its CTAs may be scheduled while the previous kernel in the stream finishes (they wait
// for it before reading anything), which hides the launch gap between back-to-back
// rotations (measured: fwd+bwd step -0.7 % on 65,536 tokens, -4 % on 16,384, -9 % on
// 7,714).
template <int D, bool LONG, int U>
cudaError_t launch_tile(const RopeArgs &a, int grid, size_t smem, cudaStream_t stream, bool pdl)
{
    if (!pdl) {
        rope_qk_tile_kernel<D, LONG, U><<<grid, kThreads, smem, stream>>>(a);
        return cudaGetLastError();
    }
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, rope_qk_tile_kernel<D, LONG, U>, a);
}

// The generic head_dim instance keeps 2 pair units per thread.
template <bool LONG, int U>
cudaError_t dispatch_dim(const RopeArgs &a, int grid, size_t smem, cudaStream_t stream, bool pdl)
{
    switch (a.head_dim) {
    case 64: return launch_tile<64, LONG, U>(a, grid, smem, stream, pdl);
    case 96: return launch_tile<96, LONG, U>(a, grid, smem, stream, pdl);
    case 128: return launch_tile<128, LONG, U>(a, grid, smem, stream, pdl);
    case 256: return launch_tile<256, LONG, U>(a, grid, smem, stream, pdl);
    default: return launch_tile<0, LONG, 2>(a, grid, smem, stream, pdl);
    }
}

// A strided bf16 view of `rows` x `heads` blocks of head_dim contiguous elements.
struct View {
    const void *base;
    int64_t rows, heads, ts, hs, d;

    int64_t span_elems() const { return (rows - 1) * ts + (heads - 1) * hs + d; }
    int64_t bytes() const { return span_elems() * 2; }
};

// Distinct (row, head) pairs address disjoint blocks: with the two dimensions sorted by
// stride, the smaller stride covers a block and the larger one covers every block of
// the smaller dimension.  A dimension of extent 1 is ignored.
bool view_injective(const View &v)
{
    int64_t s1 = v.ts, n1 = v.rows, s2 = v.hs, n2 = v.heads;
    if (n1 <= 1) { s1 = s2; n1 = n2; s2 = 0; n2 = 1; }
    if (n2 > 1 && s2 < s1) { std::swap(s1, s2); std::swap(n1, n2); }
    if (n1 > 1 && s1 < v.d) return false;
    if (n2 > 1 && s2 < n1 * s1) return false;
    return true;
}

// Two views share no element.  True when their address ranges are disjoint, or when
// both step tokens by the same stride S, each token's block fits in S, and the second
// view's block sits after the first's inside every period of S (the Q and K slices of
// a fused QKV projection output).
bool views_disjoint(const View &a, const View &b)
{
    if (!overlap(a.base, a.bytes(), b.base, b.bytes())) return true;
    if (a.rows != b.rows || a.ts != b.ts || a.ts <= 0 || a.rows < 1) return false;
    const int64_t S = a.ts;
    const int64_t ea = (a.heads - 1) * a.hs + a.d;
    const int64_t eb = (b.heads - 1) * b.hs + b.d;
    if (ea > S || eb > S) return false;
    const int64_t delta_bytes = static_cast<int64_t>(reinterpret_cast<uintptr_t>(b.base)) -
                                static_cast<int64_t>(reinterpret_cast<uintptr_t>(a.base));
    if (delta_bytes % 2 != 0) return false;
    const int64_t r = ((delta_bytes / 2) % S + S) % S;
    return r >= ea && r + eb <= S;
}

// The view's span in elements, computed without wrapping, stays below 2^56 (so that
// the int64 span, byte counts and overlap tests below cannot overflow).
bool span_fits(const View &v)
{
    const __int128 span = static_cast<__int128>(v.rows - 1) * v.ts + static_cast<__int128>(v.heads - 1) * v.hs + v.d;
    return span < (static_cast<__int128>(1) << 56);
}

int check_view(const View &v)
{
    if (v.base == nullptr) return ROPE_ERR_NULL;
    if (!aligned(v.base, 16) || v.ts % 8 != 0 || v.hs % 8 != 0) return ROPE_ERR_ALIGN;
    if (v.ts < 0 || v.hs < 0 || !span_fits(v)) return ROPE_ERR_SHAPE;
    if (!view_injective(v)) return ROPE_ERR_OVERLAP;
    return ROPE_OK;
}

// Check word of a cache descriptor: FNV-1a (64-bit) over the bytes of every other
// field, so that a descriptor not written by the build, or changed after it, is caught.
uint64_t cache_check_word(const rope_cos_sin_cache &c)
{
    uint64_t h = 1469598103934665603ull;
    auto mix = [&h](const void *p, size_t n) {
        const unsigned char *b = static_cast<const unsigned char *>(p);
        for (size_t i = 0; i < n; ++i) {
            h ^= b[i];
            h *= 1099511628211ull;
        }
    };
    const uintptr_t data = reinterpret_cast<uintptr_t>(c.data);
    mix(&data, sizeof data);
    mix(&c.rows, sizeof c.rows);
    mix(&c.head_dim, sizeof c.head_dim);
    mix(&c.device, sizeof c.device);
    mix(&c.theta, sizeof c.theta);
    mix(&c.position_scale, sizeof c.position_scale);
    return h;
}

// The cache serves this rotation: written by the build, for the same head_dim, theta
// and position_scale, with a table inside the limits the build enforces.
int check_cache(const rope_cos_sin_cache *c, int32_t head_dim, double theta, double scale)
{
    if (c == nullptr) return ROPE_OK;
    if (c->check != cache_check_word(*c)) return ROPE_ERR_CACHE;
    if (c->head_dim != head_dim || !(c->theta == theta) || !(c->position_scale == scale)) return ROPE_ERR_CACHE;
    if (c->rows < 0 || c->rows > kMaxTokens || (c->rows > 0 && c->data == nullptr)) return ROPE_ERR_CACHE;
    if (c->data != nullptr && !aligned(c->data, 16)) return ROPE_ERR_ALIGN;
    return ROPE_OK;
}

// A cache with rows is read by kernels of the current device only.
int check_cache_device(const rope_cos_sin_cache *c)
{
    if (c == nullptr || c->rows == 0) return ROPE_OK;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return ROPE_ERR_LAUNCH;
    return dev == c->device ? ROPE_OK : ROPE_ERR_CACHE;
}

}  // namespace

// Every check of a descriptor that does not depend on where Q and K live: sizes, flags,
// theta and scale, the position source (cu_seqlens with an offset or segments, or
// position ids) and the cache.  Shared by rope_qk_apply and the host-buffer entry
// points, which run it on the whole pack before they copy anything.  No CUDA call.
int rope_qk_check_pack(const rope_qk_desc *dp)
{
    if (dp == nullptr) return ROPE_ERR_NULL;
    const rope_qk_desc &p = *dp;
    const int64_t T = p.total_tokens;
    if (T < 0 || p.n_seqs < 0 || p.n_q_heads < 1 || p.n_kv_heads < 1 || p.token_offset < 0 ||
        p.n_segments < 0 || p.n_segments > kMaxSegments)
        return ROPE_ERR_SHAPE;
    if (p.n_q_heads > (1 << 20) || p.n_kv_heads > (1 << 20)) return ROPE_ERR_SHAPE;
    if ((p.flags & ~ROPE_FLAG_POSITION_IDS_INT64) != 0 || p.reserved != 0) return ROPE_ERR_UNSUPPORTED;
    int rc = check_head_dim(p.head_dim);
    if (rc != ROPE_OK) return rc;
    if ((rc = check_theta(p.theta)) != ROPE_OK) return rc;
    if ((rc = check_scale(p.position_scale)) != ROPE_OK) return rc;
    if (T == 0) return ROPE_OK;     // nothing is read or written; pointers may be NULL
    const bool ids64 = (p.flags & ROPE_FLAG_POSITION_IDS_INT64) != 0;
    if (p.position_ids != nullptr) {
        if (p.n_segments > 0) return ROPE_ERR_UNSUPPORTED;
        if (ids64 && !aligned(p.position_ids, 8)) return ROPE_ERR_ALIGN;
    } else {
        // positions must stay exact in binary32: global token indices below 2^24
        // (explicit position ids outside [0, 2^24) are skipped by the kernel instead)
        if (p.cu_seqlens == nullptr) return ROPE_ERR_NULL;
        if (p.n_segments == 0) {
            if (p.token_offset + T > kMaxTokens) return ROPE_ERR_UNSUPPORTED;
        } else {
            if (p.segments == nullptr) return ROPE_ERR_NULL;
            if (p.token_offset != 0 || p.segments[0].row_start != 0) return ROPE_ERR_SHAPE;
            for (int i = 0; i < p.n_segments; ++i) {
                const rope_qk_segment &g = p.segments[i];
                const int64_t end = i + 1 < p.n_segments ? p.segments[i + 1].row_start : T;
                if (g.row_start >= end || end > T || g.token_start < 0) return ROPE_ERR_SHAPE;
                if (g.token_start > kMaxTokens || end - g.row_start > kMaxTokens - g.token_start)
                    return ROPE_ERR_UNSUPPORTED;
            }
        }
    }
    return check_cache(p.cos_sin_cache, p.head_dim, p.theta, p.position_scale);
}

namespace {

// What rope_qk_apply launches for a descriptor: the kernel's arguments, grid, shared
// memory and instance (head_dim template, 0 = generic; 64-bit offsets or not).
struct Launch {
    RopeArgs a;
    int grid = 0;
    size_t smem = 0;
    int d_instance = 0;
    int unroll = 2;
    bool long_index = false;
};

int instance_for(int head_dim)
{
    switch (head_dim) {
    case 64: case 96: case 128: case 256: return head_dim;
    default: return 0;
    }
}

// Every argument check of rope_qk_apply, then the launch plan.  With `check_device`,
// also the cache's device (the one CUDA runtime call of the checks).  For T == 0
// returns ROPE_OK with L->grid == 0 (nothing to launch).
int plan_rotation(const rope_qk_desc *dp, Launch *L, bool check_device)
{
    int rc = rope_qk_check_pack(dp);
    if (rc != ROPE_OK) return rc;
    const rope_qk_desc &p = *dp;
    const int64_t T = p.total_tokens;
    L->grid = 0;
    if (T == 0) return ROPE_OK;
    if (T > INT32_MAX / 2) return ROPE_ERR_UNSUPPORTED;
    const bool ids64 = (p.flags & ROPE_FLAG_POSITION_IDS_INT64) != 0;

    const int64_t d = p.head_dim;
    const View q{p.q, T, p.n_q_heads, p.q_stride_token, p.q_stride_head, d};
    const View k{p.k, T, p.n_kv_heads, p.k_stride_token, p.k_stride_head, d};
    const bool in_place = p.q_out == nullptr && p.k_out == nullptr;
    if (!in_place && (p.q_out == nullptr || p.k_out == nullptr)) return ROPE_ERR_NULL;
    const View qo = in_place ? q : View{p.q_out, T, p.n_q_heads, p.q_out_stride_token, p.q_out_stride_head, d};
    const View ko = in_place ? k : View{p.k_out, T, p.n_kv_heads, p.k_out_stride_token, p.k_out_stride_head, d};
    for (const View *v : {&q, &k, &qo, &ko})
        if ((rc = check_view(*v)) != ROPE_OK) return rc;
    if (!views_disjoint(q, k)) return ROPE_ERR_OVERLAP;
    if (!in_place) {
        if (!views_disjoint(qo, ko)) return ROPE_ERR_OVERLAP;
        for (const View *o : {&qo, &ko})
            for (const View *i : {&q, &k})
                if (overlap(o->base, o->bytes(), i->base, i->bytes())) return ROPE_ERR_OVERLAP;
    }
    if (check_device && (rc = check_cache_device(p.cos_sin_cache)) != ROPE_OK) return rc;

    RopeArgs &a = L->a;
    a = RopeArgs{};
    a.q_in = static_cast<const __nv_bfloat16 *>(p.q);
    a.k_in = static_cast<const __nv_bfloat16 *>(p.k);
    a.q_out = static_cast<__nv_bfloat16 *>(const_cast<void *>(qo.base));
    a.k_out = static_cast<__nv_bfloat16 *>(const_cast<void *>(ko.base));
    a.q_ts = q.ts;  a.q_hs = q.hs;  a.k_ts = k.ts;  a.k_hs = k.hs;
    a.qo_ts = qo.ts; a.qo_hs = qo.hs; a.ko_ts = ko.ts; a.ko_hs = ko.hs;
    const bool ids = p.position_ids != nullptr;
    a.cu = p.cu_seqlens;
    a.pos_ids = ids && !ids64 ? p.position_ids : nullptr;
    a.pos_ids64 = ids && ids64 ? reinterpret_cast<const long long *>(p.position_ids) : nullptr;
    a.seq_used = ids ? nullptr : p.seq_used;
    const rope_cos_sin_cache *cache = p.cos_sin_cache;
    a.cache = cache != nullptr && cache->rows > 0 ? reinterpret_cast<const float4 *>(cache->data) : nullptr;
    a.cache_rows = a.cache != nullptr ? static_cast<int32_t>(cache->rows) : 0;
    a.n_seqs = ids ? 0 : p.n_seqs;
    a.stage_cu = !ids && p.n_seqs < kMaxStagedCu ? 1 : 0;
    a.n_tokens = static_cast<int32_t>(T);
    // row r of segment i is token r + seg_delta[i] of cu_seqlens' stream (all below 2^24)
    if (ids || p.n_segments == 0) {
        a.n_seg = 1;
        a.seg_row[0] = 0;
        a.seg_delta[0] = ids ? 0 : static_cast<int32_t>(p.token_offset);
    } else {
        a.n_seg = p.n_segments;
        for (int i = 0; i < p.n_segments; ++i) {
            a.seg_row[i] = static_cast<int32_t>(p.segments[i].row_start);
            a.seg_delta[i] = static_cast<int32_t>(p.segments[i].token_start - p.segments[i].row_start);
        }
    }
    a.hq = p.n_q_heads;
    a.hkv = p.n_kv_heads;
    a.h_tot = p.n_q_heads + p.n_kv_heads;
    a.head_dim = p.head_dim;
    a.tile_tokens = pick_tile_tokens(a.h_tot, p.head_dim, a.seq_used != nullptr ? kTileUnitsSeqUsed : kTileUnits);
    if (a.cache != nullptr && a.seq_used == nullptr) {
        const int half = pick_tile_tokens(a.h_tot, p.head_dim, kTileUnitsCached);
        if ((T + half - 1) / half < kWideGrid) a.tile_tokens = half;
    }
    a.in_place = in_place ? 1 : 0;
    a.bwd = p.backward ? 1 : 0;
    a.div_htot = make_fastdiv(static_cast<uint32_t>(a.h_tot));
    a.div_cph = make_fastdiv(static_cast<uint32_t>(p.head_dim / 16));
    host_inv_freq(p.theta, p.head_dim, p.position_scale, a.w);

    L->grid = static_cast<int>((T + a.tile_tokens - 1) / a.tile_tokens);
    // 4*cph float4 of (cos, sin) per token, then the staged cu_seqlens
    L->smem = static_cast<size_t>(a.tile_tokens) * (p.head_dim / 2) * sizeof(float2) +
              (a.stage_cu ? static_cast<size_t>(a.n_seqs + 1) * sizeof(int32_t) : 0);
    // 64-bit offsets only when some element offset of a view reaches 2^31
    L->long_index = false;
    for (const View *v : {&q, &k, &qo, &ko})
        L->long_index = L->long_index || v->span_elems() > INT32_MAX;
    L->d_instance = instance_for(p.head_dim);
    // Pair units in flight per thread: 4 for large launches with 32-bit offsets that read
    // their cos/sin from a cache (the tile's first batch then covers most of a wide
    // token's units before the position search); 3 for smaller such launches whose tile
    // fits in one batch of 3 (the whole tile then streams in one round trip: 1-token
    // tiles on 40 heads of 128, 0.7-1.5 % faster than 2), and for launches with 64-bit
    // offsets that read a cache (72 registers; 2^20 tokens on 40 heads of 128: 3,095
    // against 3,121 us with 2, where 4 was slower); 2 otherwise (more resident CTAs, a
    // cheaper evaluation of cos/sin in the kernel); the generic head_dim instance always 2.
    const bool cached = a.cache != nullptr && L->d_instance != 0;
    const int tile_units = a.tile_tokens * a.h_tot * (p.head_dim / 16);
    if (cached && !L->long_index && L->grid >= kWideGrid)
        L->unroll = 4;
    else if (cached && !L->long_index && a.seq_used == nullptr && tile_units <= 3 * kThreads)
        L->unroll = 3;
    else if (cached && L->long_index && a.seq_used == nullptr)
        L->unroll = 3;
    else
        L->unroll = 2;
    return ROPE_OK;
}

int rope_qk_apply_impl(const rope_qk_desc *dp, void *stream, bool pdl)
{
    Launch L;
    const int rc = plan_rotation(dp, &L, true);
    if (rc != ROPE_OK || L.grid == 0) return rc;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t err;
    if (L.unroll == 4)
        err = dispatch_dim<false, 4>(L.a, L.grid, L.smem, s, pdl);
    else if (L.unroll == 3)
        err = L.long_index ? dispatch_dim<true, 3>(L.a, L.grid, L.smem, s, pdl)
                           : dispatch_dim<false, 3>(L.a, L.grid, L.smem, s, pdl);
    else
        err = L.long_index ? dispatch_dim<true, 2>(L.a, L.grid, L.smem, s, pdl)
                           : dispatch_dim<false, 2>(L.a, L.grid, L.smem, s, pdl);
    return err == cudaSuccess ? ROPE_OK : ROPE_ERR_LAUNCH;
}

// The contiguous [T, H, d] form of the two simple entry points.
int rope_qk_run(void *q, void *k, const int32_t *cu_seqlens, int32_t n_seqs, int64_t total_tokens,
                int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim, double theta,
                int32_t in_place, void *q_out, void *k_out, const rope_cos_sin_cache *cache,
                void *stream, int bwd)
{
    if (total_tokens < 0 || n_seqs < 0 || n_q_heads < 1 || n_kv_heads < 1) return ROPE_ERR_SHAPE;
    // out of place needs both outputs (a desc with no outputs would mean in place)
    if (total_tokens > 0 && !in_place && (q_out == nullptr || k_out == nullptr)) return ROPE_ERR_NULL;
    rope_qk_desc p{};
    const int64_t hqd = static_cast<int64_t>(n_q_heads) * head_dim;
    const int64_t hkd = static_cast<int64_t>(n_kv_heads) * head_dim;
    p.q = q;  p.q_stride_token = hqd; p.q_stride_head = head_dim;
    p.k = k;  p.k_stride_token = hkd; p.k_stride_head = head_dim;
    if (!in_place) {
        p.q_out = q_out; p.q_out_stride_token = hqd; p.q_out_stride_head = head_dim;
        p.k_out = k_out; p.k_out_stride_token = hkd; p.k_out_stride_head = head_dim;
    }
    p.cu_seqlens = cu_seqlens;
    p.n_seqs = n_seqs;
    p.total_tokens = total_tokens;
    p.n_q_heads = n_q_heads;
    p.n_kv_heads = n_kv_heads;
    p.head_dim = head_dim;
    p.backward = bwd;
    p.theta = theta;
    p.position_scale = 1.0;
    p.cos_sin_cache = cache;
    return rope_qk_apply_impl(&p, stream, true);
}

}  // namespace

// rope_qk_apply with plain launches, for the host-buffer pipeline (its rotations follow
// cross-stream event waits, where an overlapped launch has nothing to hide).
int rope_qk_apply_plain_launch(const rope_qk_desc *desc, void *stream)
{
    return rope_qk_apply_impl(desc, stream, false);
}

extern "C" {

int rope_qk_fwd(void *q, void *k, const int32_t *cu_seqlens, int32_t n_seqs, int64_t total_tokens,
                int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim, double theta,
                int32_t in_place, void *q_out, void *k_out, const rope_cos_sin_cache *cos_sin_cache,
                void *stream)
{
    return rope_qk_run(q, k, cu_seqlens, n_seqs, total_tokens, n_q_heads, n_kv_heads, head_dim,
                       theta, in_place, q_out, k_out, cos_sin_cache, stream, 0);
}

int rope_qk_bwd(void *q, void *k, const int32_t *cu_seqlens, int32_t n_seqs, int64_t total_tokens,
                int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim, double theta,
                int32_t in_place, void *q_out, void *k_out, const rope_cos_sin_cache *cos_sin_cache,
                void *stream)
{
    return rope_qk_run(q, k, cu_seqlens, n_seqs, total_tokens, n_q_heads, n_kv_heads, head_dim,
                       theta, in_place, q_out, k_out, cos_sin_cache, stream, 1);
}

int64_t rope_cos_sin_cache_bytes(int64_t cache_rows, int32_t head_dim)
{
    if (cache_rows < 0 || check_head_dim(head_dim) != ROPE_OK) return -1;
    return cache_rows * head_dim * static_cast<int64_t>(sizeof(float));
}

int rope_cos_sin_cache_build(rope_cos_sin_cache *cache, float *data, int64_t rows, int32_t head_dim,
                             double theta, double position_scale, void *stream)
{
    if (cache == nullptr) return ROPE_ERR_NULL;
    if (rows < 0) return ROPE_ERR_SHAPE;
    int rc = check_head_dim(head_dim);
    if (rc != ROPE_OK) return rc;
    if ((rc = check_theta(theta)) != ROPE_OK) return rc;
    if ((rc = check_scale(position_scale)) != ROPE_OK) return rc;
    if (rows > kMaxTokens) return ROPE_ERR_UNSUPPORTED;
    rope_cos_sin_cache c{};
    c.data = data;
    c.rows = rows;
    c.head_dim = head_dim;
    c.device = -1;                  // no rows: no table to read, valid on every device
    c.theta = theta;
    c.position_scale = position_scale;
    if (rows > 0) {
        if (data == nullptr) return ROPE_ERR_NULL;
        if (!aligned(data, 16)) return ROPE_ERR_ALIGN;
        if (cudaGetDevice(&c.device) != cudaSuccess) return ROPE_ERR_LAUNCH;
        CacheArgs a{};
        host_inv_freq(theta, head_dim, position_scale, a.w);
        const int cph = head_dim / 16;
        const int64_t n = rows * 4 * cph;
        const int64_t blocks64 = (n + 255) / 256;
        const int blocks = static_cast<int>(blocks64 < 152 * 64 ? blocks64 : 152 * 64);
        cos_sin_cache_kernel<<<blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(
            reinterpret_cast<float4 *>(data), rows, cph, a);
        if (cudaGetLastError() != cudaSuccess) return ROPE_ERR_LAUNCH;
    }
    c.check = cache_check_word(c);
    *cache = c;
    return ROPE_OK;
}

int rope_qk_apply(const rope_qk_desc *desc, void *stream)
{
    return rope_qk_apply_impl(desc, stream, true);
}

int rope_qk_launch_info(const rope_qk_desc *desc, rope_qk_launch *info)
{
    if (info == nullptr) return ROPE_ERR_NULL;
    Launch L;
    const int rc = plan_rotation(desc, &L, false);
    if (rc != ROPE_OK) return rc;
    info->head_dim_instance = L.grid > 0 ? L.d_instance : 0;
    info->long_index = L.grid > 0 && L.long_index ? 1 : 0;
    info->grid = L.grid;
    info->tile_tokens = L.grid > 0 ? L.a.tile_tokens : 0;
    info->threads = L.grid > 0 ? kThreads : 0;
    info->smem_bytes = static_cast<int32_t>(L.smem);
    info->unroll = L.grid > 0 ? L.unroll : 0;
    return ROPE_OK;
}

int rope_qk_positions(const int32_t *cu_seqlens, int32_t n_seqs, int64_t total_tokens,
                      int32_t *pos_out, void *stream)
{
    if (total_tokens < 0 || n_seqs < 0) return ROPE_ERR_SHAPE;
    if (total_tokens > kMaxTokens) return ROPE_ERR_UNSUPPORTED;
    if (total_tokens == 0) return ROPE_OK;
    if (cu_seqlens == nullptr || pos_out == nullptr) return ROPE_ERR_NULL;
    const int n = static_cast<int>(total_tokens);
    const int blocks = (n + 255) / 256 < 152 * 16 ? (n + 255) / 256 : 152 * 16;
    positions_kernel<<<blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(cu_seqlens, n_seqs, n, pos_out);
    return cudaGetLastError() == cudaSuccess ? ROPE_OK : ROPE_ERR_LAUNCH;
}

int rope_validate_cu_seqlens(const int32_t *cu_seqlens, int32_t n_seqs, int64_t total_tokens,
                             int32_t *err_word, void *stream)
{
    if (total_tokens < 0 || n_seqs < 0) return ROPE_ERR_SHAPE;
    if (cu_seqlens == nullptr || err_word == nullptr) return ROPE_ERR_NULL;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(err_word, 0, sizeof(int32_t), s) != cudaSuccess) return ROPE_ERR_LAUNCH;
    const int64_t blocks64 = (static_cast<int64_t>(n_seqs) + 255) / 256;
    const int blocks = static_cast<int>(blocks64 < 1 ? 1 : (blocks64 < 152 * 16 ? blocks64 : 152 * 16));
    validate_kernel<<<blocks, 256, 0, s>>>(cu_seqlens, n_seqs, total_tokens, err_word);
    return cudaGetLastError() == cudaSuccess ? ROPE_OK : ROPE_ERR_LAUNCH;
}

int rope_cos_sin_eval(const float *phi, float *cos_out, float *sin_out, int64_t n, int32_t mode, void *stream)
{
    if (n < 0) return ROPE_ERR_SHAPE;
    if (mode < ROPE_COS_SIN_AS_ROTATION || mode > ROPE_COS_SIN_BINARY32_ONLY) return ROPE_ERR_KIND;
    if (n == 0) return ROPE_OK;
    if (phi == nullptr || cos_out == nullptr || sin_out == nullptr) return ROPE_ERR_NULL;
    const int64_t blocks64 = (n + 255) / 256;
    const int blocks = static_cast<int>(blocks64 < 152 * 32 ? blocks64 : 152 * 32);
    cos_sin_eval_kernel<<<blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(phi, cos_out, sin_out, n, mode);
    return cudaGetLastError() == cudaSuccess ? ROPE_OK : ROPE_ERR_LAUNCH;
}

int rope_qk_inv_freq(double theta, int32_t head_dim, double position_scale, float *w_out)
{
    int rc = check_head_dim(head_dim);
    if (rc != ROPE_OK) return rc;
    if ((rc = check_theta(theta)) != ROPE_OK) return rc;
    if ((rc = check_scale(position_scale)) != ROPE_OK) return rc;
    if (w_out == nullptr) return ROPE_ERR_NULL;
    host_inv_freq(theta, head_dim, position_scale, w_out);
    return ROPE_OK;
}

const char *rope_strerror(int status)
{
    switch (status) {
    case ROPE_OK: return "ok";
    case ROPE_ERR_NULL: return "a required pointer is NULL";
    case ROPE_ERR_SHAPE: return "invalid size, stride or segment list: negative count/stride/offset, head count < 1, "
                                "segments not starting at row 0 or not increasing";
    case ROPE_ERR_HEAD_DIM: return "head_dim must be a multiple of 16 in [16, 256]";
    case ROPE_ERR_ALIGN: return "Q/K/outputs and the cos/sin cache must be 16-byte aligned (int64 position ids 8-byte), "
                                "strides multiples of 8 elements";
    case ROPE_ERR_OVERLAP: return "Q and K overlap, a view overlaps itself, or an output overlaps an input";
    case ROPE_ERR_UNSUPPORTED: return "unsupported: a global token index or cache row beyond 2^24 (exact fp32 positions), "
                                      "an unknown flag bit, segments with position ids, or a workspace below 8 tokens";
    case ROPE_ERR_LAUNCH: return "the CUDA runtime rejected a launch";
    case ROPE_ERR_THETA: return "theta and position_scale must be finite and > 0";
    case ROPE_ERR_KIND: return "unknown activation kind";
    case ROPE_ERR_WORKSPACE: return "one token's Q and K rows exceed the 32 MiB static staging array";
    case ROPE_ERR_CACHE: return "the cos/sin cache was built for another theta, head_dim, position_scale or device, "
                                "or its descriptor was not written by rope_cos_sin_cache_build";
    default: return "unknown rope status";
    }
}

int rope_qk_abi_version(void) { return ROPE_QK_ABI_VERSION; }

}  // extern "C"
