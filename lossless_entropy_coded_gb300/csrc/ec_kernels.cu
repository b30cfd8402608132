/*
 * ec_kernels.cu -- sm_103a kernels and the device-side entry points of the C ABI
 * (ec_decode, ec_decode_batch, ec_gemv, ec_gemv_group, ec_bf16_gemv, ec_status).
 *
 * Huffman path (DFloat11, "70% Size, 100% Accuracy", Algorithm 1, re-cut for the
 * fused product of MINE section 4 "Fused mvm"):
 *   one warp owns one tile of 32 * steps weights.  Each lane decodes its own
 *   codeword sequence (positions l, l + 32, ...) from a byte offset stored in the
 *   tile record, with a 12-bit level-1 table in shared memory and 8-bit
 *   sub-tables behind pointer entries (the hierarchical LUTs of Fig. 4 / 14).
 *   Decoded exponent fields go to a per-warp shared-memory stage, 1024 weights at
 *   a time; the stage is then read back 8 consecutive weights per lane and merged
 *   with the raw sign/mantissa bytes:
 *       bf16 = (sign << 15) | (exponent << 7) | mantissa      (Algorithm 1 / Eq. (1))
 *   and either stored (decode) or multiplied with x in FP32 (GEMV).  Partial sums
 *   of a row are reduced across the warp with shuffles and written once, or added
 *   atomically when a row spans several tiles.
 *
 * rANS path (EntroPack section 3.6, appendix C.3): one warp per tile, lane l
 * decodes positions 32 j + l; a lane whose state drops below 2^16 pulls the next
 * 16-bit word, the lanes of one step taking consecutive words in lane order
 * (ballot + popc).  w = code * scale (FP16 scale per 128 weights) is exact in FP32.
 *
 * Robustness: every loop has a fixed trip count; reads of code words, sub-tables
 * and payload words are clamped to the tile / table and an out-of-range index sets
 * the device status word (EC_ERR_CORRUPT) instead of faulting.
 */
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "ec_internal.h"

namespace {

constexpr int kWarps = 8;          /* warps per CTA (rANS and BF16 kernels) */
constexpr unsigned kFull = 0xFFFFFFFFu;
constexpr int kMaxDecodeBatch = EC_MAX_DECODE_BATCH;

/* ------------------------------------------------------------ descriptors */
struct HuffMat {
    const uint8_t* records;
    const uint32_t* tile_off;   /* 16-byte units */
    const uint32_t* table;      /* level 1 + sub-tables */
    int64_t table_words;
    float* y;                   /* GEMV output [batch, n_rows] */
    uint16_t* out;              /* decode output [n_rows, k_cols] */
    int64_t n_rows, k_cols, k_pad;
    int64_t n_tiles, tile_begin;
    int64_t records_bytes;
    int32_t steps, atomic_y;
};

struct HuffGemvArgs {
    HuffMat m[EC_MAX_GROUP];
    int count;
    int batch;
    const uint16_t* x;          /* [batch, k_cols] */
    int64_t total_tiles;
    int* status;
    int code_bytes;             /* per-warp code buffer */
    float* part;                /* allocation-free variant: per (row, tile) partial sums */
    int part_slots;             /* partial-sum slots per row */
};

struct HuffDecodeArgs {
    HuffMat m[kMaxDecodeBatch];
    int count;
    int64_t total_tiles;
    int* status;
    int code_bytes;
};

struct RansMat {
    const uint8_t* records;
    const uint32_t* tile_off;
    const uint32_t* table;      /* 2^prob_bits slot entries */
    const uint16_t* scales;     /* [n_rows, k_pad / 128] */
    float* y;
    uint16_t* out;
    int64_t n_rows, k_cols, k_pad;
    int64_t n_tiles;
    int64_t records_bytes;
    int32_t steps, prob_bits, atomic_y, words_cap;
};

struct RansArgs {
    RansMat m;
    int batch;
    const uint16_t* x;
    int* status;
};

/* ------------------------------------------------------------ small helpers */
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}

__device__ __forceinline__ void flag_corrupt(int* status) { atomicOr(status, 1); }

/* Which matrix of a launch owns combined tile index g (count is small). */
template <class Args>
__device__ __forceinline__ int owner(const Args& a, int64_t g) {
    int k = 0;
    while (k + 1 < a.count && g >= a.m[k + 1].tile_begin) ++k;
    return k;
}

/* Start and length (bytes) of tile t's record; a range outside the records region
 * (only possible with a corrupted offset table) yields an empty record. */
__device__ __forceinline__ int64_t record_span(const uint32_t* __restrict__ tile_off, int64_t t, int64_t records_bytes,
                                               int64_t* bytes, int* status, int lane) {
    const int64_t a = (int64_t)__ldg(tile_off + t) * 16, b = (int64_t)__ldg(tile_off + t + 1) * 16;
    if (a > b || b > records_bytes) {
        if (lane == 0) flag_corrupt(status);
        *bytes = 0;
        return 0;
    }
    *bytes = b - a;
    return a;
}

/* Copy `bytes` (multiple of 16) from global to shared memory with the warp. */
__device__ __forceinline__ void warp_copy16(void* dst, const void* src, int bytes, int lane) {
    const uint4* s = (const uint4*)src;
    uint4* d = (uint4*)dst;
    for (int i = lane; i < bytes / 16; i += 32) d[i] = __ldg(s + i);
}

/* floor(t * T / kp) where `unit` divides both T and kp (32-bit division when it fits). */
__device__ __forceinline__ int64_t tile_row(int64_t t, int64_t T, int64_t kp, int64_t unit) {
    const uint64_t a = (uint64_t)t * (uint64_t)(T / unit), b = (uint64_t)(kp / unit);
    if (a < 0xFFFFFFFFull && b < 0xFFFFFFFFull) return (int64_t)((uint32_t)a / (uint32_t)b);
    return (int64_t)(a / b);
}

/* ============================================================ Huffman path */
/*
 * Work layout.  One warp decodes one tile at a time; lane l owns the tile's
 * symbols i = 0 .. S-1 at positions 32 i + l and, unlike a DFloat11 thread that
 * hands its output to a block-wide write buffer, lane l also multiplies them:
 * exponents go to a lane-private byte stage in shared memory (two buffers of
 * kC symbols + spill, lane stride kLane = 11 words so the 32 lanes' stores and
 * 4-byte reads fall in distinct banks), the matching raw bytes arrive
 * lane-transposed with one 16-byte load per 16 symbols, and x is kept transposed
 * in shared memory (xs_t[l][j] = x[32 j + l]) so lane l finds x for its symbols
 * contiguously.  Decoding chunk c + 1 is interleaved with the multiply-accumulate
 * of chunk c.
 */
constexpr int kHW = 24;                        /* max warps per CTA */
constexpr int kC = 32;                         /* symbols per lane per chunk */
constexpr int kLane = 44;                      /* stage bytes per lane per buffer (11 words) */
constexpr int kStageBuf = 32 * kLane;          /* one buffer of the warp */
constexpr int kStageBytes = 2 * kStageBuf;     /* two buffers */
constexpr int kSlackPairs = 32;                /* zero pairs after the code area (even) */
constexpr uint32_t kMultiBytes = 4u * EC_MULTI_WORDS;
static_assert(kLane >= kC + 8 && kLane % 4 == 0 && (kLane / 4) % 2 == 1, "stage lane stride");

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ uint2 lds64(uint32_t a) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a) : "memory");
    return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
    return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a) : "memory");
    return v;
}
__device__ __forceinline__ void sts8(uint32_t a, uint32_t v) {
    asm volatile("st.shared.u8 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}
__device__ __forceinline__ void sts16(uint32_t a, uint32_t v) {
    asm volatile("st.shared.u16 [%0], %1;" ::"r"(a), "h"((unsigned short)v) : "memory");
}
__device__ __forceinline__ void sts32(uint32_t a, uint32_t v) {
    asm volatile("st.shared.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}

/* Codeword longer than the level-1 window (rare): walk the hierarchical table in
 * global memory from its level-1 entry for this window.  Returns the exponent with
 * a count of 1 in the multi-entry layout (.x) and the codeword length (.y, up to
 * 24 bits, which the 4-bit length field of a multi entry cannot hold).  Corrupt
 * data (no codeword matches) yields exponent 0 of length 1 and sets the status. */
__device__ __noinline__ uint2 long_codeword(uint32_t win, const uint32_t* __restrict__ hier, int64_t hier_words,
                                            int* status) {
    uint32_t ent = __ldg(hier + (win >> (32 - EC_L1_BITS)));
#pragma unroll 1
    for (int lvl = 0; lvl < 3 && (ent & EC_ENT_PTR) && !(ent & EC_ENT_BAD); ++lvl) {
        const int used = (int)((ent >> 16) & 31);
        const int64_t at = (int64_t(1) << EC_L1_BITS) + (int64_t)(ent & 0xFFFFu) * 256 + ((win << used) >> 24);
        if (used > 24 || at >= hier_words) {
            ent = EC_ENT_BAD;
            break;
        }
        ent = __ldg(hier + at);
    }
    if (ent & (EC_ENT_PTR | EC_ENT_BAD)) {
        flag_corrupt(status);
        ent = 1u << 16;
    }
    return make_uint2(((ent & 0xFFFFu) >> 7) | (1u << 24), (ent >> 16) & 31);
}

/* Copy a tile's code area (nw words, global) into shared memory as overlapping
 * word pairs pairs[k] = (area[k], area[k + 1]), so the 64-bit window at any word is
 * one aligned 8-byte load, followed by kSlackPairs zero pairs. */
__device__ __forceinline__ void stage_pairs(uint2* pairs, const uint32_t* __restrict__ area, int nw, int lane) {
    const uint4* a4 = (const uint4*)area;
    for (int g = lane; 4 * g < nw; g += 32) {
        const uint4 a = __ldg(a4 + g);
        const uint32_t nx = 4 * g + 4 < nw ? __ldg(area + 4 * g + 4) : 0u;
        uint4* d = (uint4*)(pairs + 4 * g);
        d[0] = make_uint4(a.x, a.y, a.y, a.z);
        d[1] = make_uint4(a.z, a.w, a.w, nx);
    }
    for (int k = lane; k < kSlackPairs; k += 32) pairs[nw + k] = make_uint2(0u, 0u);
}

/* One lane's decoder: bit position p in the staged code area and the shared
 * address q of its next exponent byte. */
struct HuffLane {
    uint32_t p, q;
};

/* One multi-symbol lookup: store the entry's three exponent bytes at q, q+1, q+2 and
 * advance by the codewords it holds. */
__device__ __forceinline__ void huff_step(HuffLane& L, uint32_t l1s, uint32_t ps, const uint32_t* __restrict__ hier,
                                          int64_t hier_words, int* status) {
    const uint2 wp = lds64(ps + ((L.p >> 5) << 3));
    const uint32_t win = __funnelshift_l(wp.y, wp.x, L.p);
    uint32_t e = lds32(l1s + ((win >> (32 - EC_L1_BITS)) << 2));
    uint32_t adv = e >> 28;
    if (__builtin_expect(e < (1u << 28), 0)) {
        const uint2 lc = long_codeword(win, hier, hier_words, status);
        e = lc.x;
        adv = lc.y;
    }
    sts8(L.q, e);
    sts8(L.q + 1, e >> 8);
    sts8(L.q + 2, e >> 16);
    L.p += adv;
    L.q += (e >> 24) & 3u;
}

/* Two BF16 weights [w1 | w0] from exponent bytes (a, a+1 of e, spread by esel) and
 * raw bytes (a, a+1 of r, duplicated by rsel):
 *     w = (sign << 15) | (exponent << 7) | mantissa. */
__device__ __forceinline__ uint32_t merge_pair(uint32_t e, uint32_t esel, uint32_t r, uint32_t rsel) {
    const uint32_t spread = __byte_perm(e, 0, esel); /* [0 e1 0 e0] */
    const uint32_t dup = __byte_perm(r, 0, rsel);    /* [r1 r1 r0 r0] */
    return spread * 128u + (dup & 0x807F807Fu);      /* fields do not overlap: + is | */
}

/* Eight weights: exponent bytes e = (e0..e3, e4..e7), raw bytes r0 (4), r1 (4). */
__device__ __forceinline__ void merge8(uint2 e, uint32_t r0, uint32_t r1, uint32_t (&w)[4]) {
    w[0] = merge_pair(e.x, 0x4140, r0, 0x1100);
    w[1] = merge_pair(e.x, 0x4342, r0, 0x3322);
    w[2] = merge_pair(e.y, 0x4140, r1, 0x1100);
    w[3] = merge_pair(e.y, 0x4342, r1, 0x3322);
}

/* acc += w0 * x0 + w1 * x1 for BF16 pairs w = [w1|w0], x = [x1|x0]; the products are
 * exact and the sums are FP32 (round to nearest). */
__device__ __forceinline__ float fma2_bf16(uint32_t w, uint32_t x, float acc) {
    asm("{\n\t.reg .b16 wl, wh, xl, xh;\n\t"
        "mov.b32 {wl, wh}, %1;\n\t"
        "mov.b32 {xl, xh}, %2;\n\t"
        "fma.rn.f32.bf16 %0, wl, xl, %0;\n\t"
        "fma.rn.f32.bf16 %0, wh, xh, %0;\n\t}"
        : "+f"(acc)
        : "r"(w), "r"(x));
    return acc;
}

__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;"); }

/* Per-warp shared memory: stage (2 buffers x 32 lanes x kLane bytes) | code pairs +
 * slack.  Multiples of 16 bytes, so 16-byte loads and stores stay aligned. */
__host__ __device__ constexpr size_t huff_warp_bytes(int code_bytes) {
    return (size_t)kStageBytes + 2 * (size_t)((code_bytes + 15) & ~15) + 8 * (size_t)kSlackPairs;
}
static_assert(kStageBytes % 16 == 0 && (8 * kSlackPairs) % 16 == 0 && kMultiBytes % 16 == 0, "alignment");
static_assert(huff_warp_bytes(16) % 16 == 0 && huff_warp_bytes(4112) % 16 == 0, "per-warp block alignment");

/* x for the GEMV, transposed per batch row: xs_t[b][l][j] = x[b][32 j + l], lane
 * stride kp / 32 + 8 entries (the +8 spreads the lanes of a quarter-warp over
 * distinct banks for 16-byte loads). */
__host__ __device__ constexpr uint32_t xs_lane_stride(uint32_t kp) { return kp / 32 + 8; }
__host__ __device__ constexpr size_t xs_row_bytes(uint32_t kp) { return (size_t)2 * 32 * xs_lane_stride(kp); }

/* Resolve tile t of matrix M.  Returns false for a record whose offsets are
 * inconsistent (status flagged, tile skipped). */
struct TileView {
    const uint8_t* raw;
    const uint32_t* area;
    int nw, S;
    int64_t row;
    uint32_t col0;
};

template <class Args>
__device__ __forceinline__ bool tile_view(const Args& a, const HuffMat& M, int64_t t, int lane, TileView& v) {
    const int64_t kp = M.k_pad;
    const int64_t T = 32 * (int64_t)M.steps;
    const int64_t base = t * T;
    const int64_t n_t = min(T, M.n_rows * kp - base);
    int64_t rec_bytes = 0;
    const uint8_t* rec = M.records + record_span(M.tile_off, t, M.records_bytes, &rec_bytes, a.status, lane);
    const int S = (int)(n_t / 32);
    const int raw_bytes = EC_RAW_BYTES(S);
    int64_t area_bytes = rec_bytes - 64 - raw_bytes;
    if (area_bytes < 16 || area_bytes > a.code_bytes) {
        if (lane == 0) flag_corrupt(a.status);
        return false;
    }
    v.raw = rec + 64;
    v.area = (const uint32_t*)(rec + 64 + raw_bytes);
    v.nw = (int)(area_bytes / 4);
    v.S = S;
    v.row = tile_row(t, T, kp, EC_HUFF_ROW_ALIGN);
    v.col0 = (uint32_t)(base - v.row * kp);
    return true;
}

/* Lane start in bits, clamped to the code area (a corrupt start cannot move the
 * window reads past the zero slack). */
__device__ __forceinline__ uint32_t lane_start_bits(const TileView& v, int lane) {
    const uint32_t s = __ldg((const uint16_t*)(v.raw - 64) + lane);
    return 8u * min(s, (uint32_t)(4 * v.nw));
}

/* Raw bytes of lane `lane`, symbols 16 j .. 16 j + 15 (one coalesced 16-byte load). */
__device__ __forceinline__ uint4 raw16(const TileView& v, int j, int lane) {
    return __ldg((const uint4*)v.raw + (32 * j + lane));
}

/* Decode the lane's next chunk (until q reaches q_end) interleaving up to four
 * multiply-accumulate sub-steps `fma(k)` of the previous chunk. */
template <class Fma>
__device__ __forceinline__ void huff_chunk(HuffLane& L, uint32_t q_end, int subs, uint32_t l1s, uint32_t ps,
                                           const uint32_t* __restrict__ hier, int64_t hier_words, int* status,
                                           Fma&& fma) {
#pragma unroll
    for (int k = 0; k < kC / 8; ++k) {
        if (L.q < q_end) {
            huff_step(L, l1s, ps, hier, hier_words, status);
            huff_step(L, l1s, ps, hier, hier_words, status);
        }
        if (k < subs) fma(k);
    }
#pragma unroll 1
    while (L.q < q_end) {
        huff_step(L, l1s, ps, hier, hier_words, status);
        huff_step(L, l1s, ps, hier, hier_words, status);
    }
}

/* Walk one tile: the prologue decodes chunk 0; iteration c moves chunk c's spill to
 * the other buffer and decodes chunk c + 1 there while `consume(c, k, exps)` handles
 * sub-step k (8 symbols) of chunk c. */
template <class Consume>
__device__ __forceinline__ void huff_tile(const TileView& v, uint32_t l1s, uint32_t ps, uint32_t stage_lane,
                                          const uint32_t* __restrict__ hier, int64_t hier_words, int* status,
                                          int lane, Consume&& consume) {
    const uint32_t pmax = 32u * v.nw;
    HuffLane L{lane_start_bits(v, lane), stage_lane};
    const int nch = (v.S + kC - 1) / kC;
    huff_chunk(L, stage_lane + (uint32_t)min(kC, v.S), 0, l1s, ps, hier, hier_words, status, [](int) {});
    for (int c = 0; c < nch; ++c) {
        const uint32_t X = stage_lane + (c & 1) * kStageBuf, Y = stage_lane + ((c + 1) & 1) * kStageBuf;
        const int rows_c = min(kC, v.S - c * kC);
        /* spill of chunk c (bytes kC .. kC + 7 of X) becomes the start of buffer Y */
        sts32(Y, lds32(X + kC));
        sts32(Y + 4, lds32(X + kC + 4));
        L.q = L.q - X - kC + Y;
        L.p = min(L.p, pmax);
        const int next = min(kC, v.S - (c + 1) * kC); /* symbols of chunk c + 1 (<= 0: none) */
        const uint32_t q_end = next > 0 ? Y + (uint32_t)next : 0u;
        huff_chunk(L, q_end, rows_c / 8, l1s, ps, hier, hier_words, status,
                   [&](int k) { consume(c, k, make_uint2(lds32(X + 8 * k), lds32(X + 8 * k + 4))); });
    }
}

/* ======================================================== Huffman GEMV kernel */
/* kPart = false: row sums go to y (stored, or added atomically when a row spans
 * tiles).  kPart = true (allocation-free entry point): every row segment a tile
 * produces goes to its own slot of a.part, summed into y by part_reduce_kernel. */
template <int B, bool kPart = false>
__global__ void __launch_bounds__(kHW * 32, 1) huff_gemv_kernel(const __grid_constant__ HuffGemvArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t kp = (uint32_t)a.m[0].k_pad;
    const int64_t K = a.m[0].k_cols;
    const int batch = a.batch;
    const uint32_t lx = xs_lane_stride(kp);

    /* shared: multi-symbol level-1 tables | x transposed [batch][32][lx] | per warp: stage, pairs */
    uint4* l1g = (uint4*)smem;
    uint16_t* xs = (uint16_t*)(smem + (size_t)a.count * kMultiBytes);
    uint8_t* wbase = (uint8_t*)xs + (size_t)batch * xs_row_bytes(kp) + (size_t)warp * huff_warp_bytes(a.code_bytes);
    const uint32_t stage_lane = smem_u32(wbase) + lane * kLane;
    uint2* pairs = (uint2*)(wbase + kStageBytes);
    const uint32_t pairs_s = smem_u32(pairs);
    const uint32_t xs_lane = smem_u32(xs) + lane * lx * 2;

    for (int k = 0; k < a.count; ++k) {
        const uint4* src = (const uint4*)a.m[k].table;
        for (int i = threadIdx.x; i < EC_MULTI_WORDS / 4; i += blockDim.x) l1g[k * (EC_MULTI_WORDS / 4) + i] = __ldg(src + i);
    }
    grid_dep_launch();
    grid_dep_wait(); /* x and y belong to the preceding kernel in the stream from here on */
    for (int b = 0; b < batch; ++b)
        for (uint32_t c = threadIdx.x; c < kp; c += blockDim.x)
            xs[(size_t)b * 32 * lx + (c & 31) * lx + (c >> 5)] = c < K ? a.x[(int64_t)b * K + c] : (uint16_t)0;
    __syncthreads();

    const int nwarp = blockDim.x >> 5;
    const int64_t gw = (int64_t)blockIdx.x * nwarp + warp, nw = (int64_t)gridDim.x * nwarp;
    for (int64_t g = gw; g < a.total_tiles; g += nw) {
        const int mi = owner(a, g);
        const HuffMat& M = a.m[mi];
        TileView v;
        if (!tile_view(a, M, g - M.tile_begin, lane, v)) continue;
        __syncwarp();
        stage_pairs(pairs, v.area, v.nw, lane);
        __syncwarp();
        const uint32_t l1s = smem_u32(l1g + mi * (EC_MULTI_WORDS / 4));
        int64_t row = v.row;
        uint32_t jc = v.col0 / 32; /* x column block of the current sub-step */
        const uint32_t jrow = kp / 32;
        float acc[B][2];
#pragma unroll
        for (int b = 0; b < B; ++b) acc[b][0] = acc[b][1] = 0.f;
        uint4 rw[2] = {raw16(v, 0, lane), v.S > 16 ? raw16(v, 1, lane) : make_uint4(0, 0, 0, 0)};
        uint4 rn[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};

        const int64_t t_cur = g - M.tile_begin;
        auto flush = [&](int64_t r) {
            int64_t slot = 0;
            if (kPart) /* tiles before this one that also cover row r */
                slot = t_cur - (r * M.k_pad) / (32 * (int64_t)M.steps);
#pragma unroll
            for (int b = 0; b < B; ++b) {
                if (b >= batch) break;
                const float s = warp_sum(acc[b][0] + acc[b][1]);
                if (lane == 0) {
                    if (kPart) {
                        a.part[((int64_t)b * M.n_rows + r) * a.part_slots + slot] = s;
                    } else {
                        float* dst = M.y + (int64_t)b * M.n_rows + r;
                        if (M.atomic_y) atomicAdd(dst, s);
                        else *dst = s;
                    }
                }
                acc[b][0] = acc[b][1] = 0.f;
            }
        };

        huff_tile(v, l1s, pairs_s, stage_lane, M.table + EC_MULTI_WORDS, M.table_words - EC_MULTI_WORDS, a.status,
                  lane, [&](int c, int k, const uint2& e8) {
                      if (k == 0) { /* prefetch the next chunk's raw bytes */
                          const int j = 2 * (c + 1);
                          rn[0] = 16 * j < v.S ? raw16(v, j, lane) : make_uint4(0, 0, 0, 0);
                          rn[1] = 16 * (j + 1) < v.S ? raw16(v, j + 1, lane) : make_uint4(0, 0, 0, 0);
                      }
                      if (jc >= jrow) {
                          flush(row);
                          jc -= jrow;
                          ++row;
                      }
                      const uint4& r = rw[k >> 1];
                      uint32_t w[4];
                      merge8(e8, (k & 1) ? r.z : r.x, (k & 1) ? r.w : r.y, w);
                      const uint32_t xa = xs_lane + 2 * jc;
#pragma unroll
                      for (int b = 0; b < B; ++b) {
                          if (b >= batch) break;
                          const uint4 xv = lds128(xa + (uint32_t)(b * xs_row_bytes(kp)));
                          acc[b][0] = fma2_bf16(w[0], xv.x, acc[b][0]);
                          acc[b][1] = fma2_bf16(w[1], xv.y, acc[b][1]);
                          acc[b][0] = fma2_bf16(w[2], xv.z, acc[b][0]);
                          acc[b][1] = fma2_bf16(w[3], xv.w, acc[b][1]);
                      }
                      jc += 8;
                      if (k == kC / 8 - 1) {
                          rw[0] = rn[0];
                          rw[1] = rn[1];
                      }
                  });
        flush(row);
    }
}

/* ====================================================== Huffman decode kernel */
/* Each CTA owns a contiguous range of the launch's tiles; it walks the range one
 * matrix segment at a time, with that matrix's level-1 table in shared memory.
 * Lanes merge their own symbols, then the warp transposes 256 outputs through a
 * small shared buffer so the stores to out are coalesced 16-byte writes. */
__host__ __device__ constexpr size_t decode_warp_bytes(int code_bytes) { return huff_warp_bytes(code_bytes) + 512; }

__global__ void __launch_bounds__(kHW * 32, 1) huff_decode_kernel(const __grid_constant__ HuffDecodeArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint4* l1 = (uint4*)smem;
    uint8_t* wbase = smem + kMultiBytes + (size_t)warp * decode_warp_bytes(a.code_bytes);
    const uint32_t stage_lane = smem_u32(wbase) + lane * kLane;
    uint2* pairs = (uint2*)(wbase + kStageBytes);
    const uint32_t pairs_s = smem_u32(pairs), l1s = smem_u32(l1);
    const uint32_t tbuf = smem_u32(wbase + huff_warp_bytes(a.code_bytes)); /* 256 outputs */
    grid_dep_launch();
    grid_dep_wait();

    const int64_t lo = a.total_tiles * blockIdx.x / gridDim.x, hi = a.total_tiles * (blockIdx.x + 1) / gridDim.x;
    for (int64_t cur = lo; cur < hi;) {
        const int mi = owner(a, cur);
        const HuffMat& M = a.m[mi];
        const int64_t mend = min(hi, M.tile_begin + M.n_tiles);
        __syncthreads();
        const uint4* src = (const uint4*)M.table;
        for (int i = threadIdx.x; i < EC_MULTI_WORDS / 4; i += blockDim.x) l1[i] = __ldg(src + i);
        __syncthreads();
        const int64_t kp = M.k_pad, K = M.k_cols;
        const bool vec = (K % 8) == 0;
        for (int64_t g = cur + warp; g < mend; g += (blockDim.x >> 5)) {
            TileView v;
            if (!tile_view(a, M, g - M.tile_begin, lane, v)) continue;
            __syncwarp();
            stage_pairs(pairs, v.area, v.nw, lane);
            __syncwarp();
            int64_t row = v.row;
            int64_t col0 = v.col0;
            uint4 rw[2] = {raw16(v, 0, lane), v.S > 16 ? raw16(v, 1, lane) : make_uint4(0, 0, 0, 0)};
            uint4 rn[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
            huff_tile(v, l1s, pairs_s, stage_lane, M.table + EC_MULTI_WORDS, M.table_words - EC_MULTI_WORDS,
                      a.status, lane, [&](int c, int k, const uint2& e8) {
                          if (k == 0) {
                              const int j = 2 * (c + 1);
                              rn[0] = 16 * j < v.S ? raw16(v, j, lane) : make_uint4(0, 0, 0, 0);
                              rn[1] = 16 * (j + 1) < v.S ? raw16(v, j + 1, lane) : make_uint4(0, 0, 0, 0);
                          }
                          if (col0 >= kp) {
                              col0 -= kp;
                              ++row;
                          }
                          const uint4& r = rw[k >> 1];
                          uint32_t w[4];
                          merge8(e8, (k & 1) ? r.z : r.x, (k & 1) ? r.w : r.y, w);
                          /* lane's 8 outputs are positions 32 i + lane, i = 8k'..8k'+7: transpose */
                          __syncwarp();
#pragma unroll
                          for (int j = 0; j < 8; ++j) sts16(tbuf + 64 * j + 2 * lane, w[j >> 1] >> (16 * (j & 1)));
                          __syncwarp();
                          const uint4 o = lds128(tbuf + 16 * lane);
                          const int64_t col = col0 + 8 * lane;
                          uint16_t* dst = M.out + row * K + col;
                          if (vec) {
                              if (col < K) *(uint4*)dst = o;
                          } else {
                              const uint32_t ow[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
                              for (int j = 0; j < 8; ++j)
                                  if (col + j < K) dst[j] = (uint16_t)(ow[j >> 1] >> (16 * (j & 1)));
                          }
                          col0 += 256;
                          if (k == kC / 8 - 1) {
                              rw[0] = rn[0];
                              rw[1] = rn[1];
                          }
                      });
        }
        cur = mend;
    }
}

/* ============================================================ rANS kernels */
/* Decode one tile; calls sink(step, code, lane position) for every symbol. */
template <bool kGemv, int B>
__global__ void __launch_bounds__(kWarps * 32) rans_kernel(const __grid_constant__ RansArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    const RansMat& M = a.m;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t kp = M.k_pad, K = M.k_cols;
    const uint32_t mask_b = (1u << M.prob_bits) - 1;
    uint32_t* tab = (uint32_t*)smem;
    float* xs = (float*)(smem + ((size_t)4 << M.prob_bits));
    const int batch = kGemv ? a.batch : 0;
    uint16_t* words = (uint16_t*)((uint8_t*)(xs + (size_t)batch * kp) + (size_t)warp * (2 * M.words_cap));

    for (int i = threadIdx.x; i <= (int)mask_b; i += blockDim.x) tab[i] = __ldg(M.table + i);
    if (kGemv)
        for (int b = 0; b < batch; ++b)
            for (int64_t c = threadIdx.x; c < kp; c += blockDim.x)
                xs[(int64_t)b * kp + c] = c < K ? __uint_as_float((uint32_t)a.x[(int64_t)b * K + c] << 16) : 0.f;
    __syncthreads();

    const int64_t groups = kp / 128;
    const int64_t gw = (int64_t)blockIdx.x * kWarps + warp, nw = (int64_t)gridDim.x * kWarps;
    for (int64_t t = gw; t < M.n_tiles; t += nw) {
        const int64_t T = 32 * (int64_t)M.steps;
        const int64_t base = t * T;
        const int64_t n_t = min(T, M.n_rows * kp - base);
        const int S = (int)(n_t / 32);
        int64_t rec_bytes = 0;
        const uint8_t* rec = M.records + record_span(M.tile_off, t, M.records_bytes, &rec_bytes, a.status, lane);
        if (rec_bytes < 128) {
            if (lane == 0) flag_corrupt(a.status);
            continue;
        }
        int wbytes = (int)(rec_bytes - 128);
        if (wbytes < 0 || wbytes > 2 * M.words_cap) {
            if (lane == 0) flag_corrupt(a.status);
            wbytes = max(0, min(wbytes, 2 * M.words_cap));
        }
        const int nwords = wbytes / 2;
        uint32_t x = __ldg((const uint32_t*)rec + lane);
        warp_copy16(words, rec + 128, wbytes, lane);
        __syncwarp();
        int wp = 0;
        int64_t row = tile_row(t, T, kp, EC_RANS_ROW_ALIGN);
        int64_t col0 = base - row * kp; /* column of lane 0 at the current step */
        float acc[B], accg[B];
#pragma unroll
        for (int b = 0; b < B; ++b) acc[b] = accg[b] = 0.f;

        for (int j = 0; j < S; ++j) {
            const uint32_t e = tab[x & mask_b];
            const int code = (int)(e & 15u) - 8;
            x = (e >> 16) * (x >> M.prob_bits) + ((e >> 4) & 0xFFFu);
            const bool need = x < 65536u;
            const unsigned bal = __ballot_sync(kFull, need);
            if (need) {
                const int idx = wp + __popc(bal & ((1u << lane) - 1u));
                uint32_t v = 0;
                if (idx < nwords) v = words[idx];
                else flag_corrupt(a.status);
                x = (x << 16) | v;
            }
            wp += __popc(bal);
            if (col0 >= kp) {
                if (kGemv) {
#pragma unroll
                    for (int b = 0; b < B; ++b) {
                        if (b >= batch) break;
                        const float v = warp_sum(acc[b]);
                        if (lane == 0) {
                            float* dst = M.y + (int64_t)b * M.n_rows + row;
                            if (M.atomic_y) atomicAdd(dst, v);
                            else *dst = v;
                        }
                        acc[b] = 0.f;
                    }
                }
                col0 -= kp;
                ++row;
            }
            const int64_t col = col0 + lane;
            const float scale = __half2float(__ushort_as_half(__ldg(M.scales + row * groups + col0 / 128)));
            if (kGemv) {
                const float cf = (float)code;
#pragma unroll
                for (int b = 0; b < B; ++b) {
                    if (b >= batch) break;
                    accg[b] = fmaf(cf, xs[(int64_t)b * kp + col], accg[b]);
                }
                if ((j & 3) == 3) { /* 128 positions = one scale group of one row */
#pragma unroll
                    for (int b = 0; b < B; ++b) {
                        acc[b] = fmaf(accg[b], scale, acc[b]);
                        accg[b] = 0.f;
                    }
                }
            } else if (col < K) {
                M.out[row * K + col] = __bfloat16_as_ushort(__float2bfloat16_rn((float)code * scale));
            }
            col0 += 32;
        }
        if (x != 65536u) flag_corrupt(a.status); /* every lane must return to its initial state */
        if (kGemv) {
#pragma unroll
            for (int b = 0; b < B; ++b) {
                if (b >= batch) break;
                const float v = warp_sum(acc[b]);
                if (lane == 0) {
                    float* dst = M.y + (int64_t)b * M.n_rows + row;
                    if (M.atomic_y) atomicAdd(dst, v);
                    else *dst = v;
                }
            }
        }
        __syncwarp();
    }
}

/* ======================================================== BF16 GEMV comparator */
constexpr int kRowsPerWarp = 4;

template <int B>
__global__ void __launch_bounds__(kWarps * 32) bf16_gemv_kernel(const uint16_t* __restrict__ w, int64_t n_rows,
                                                                int64_t k_cols, const uint16_t* __restrict__ x,
                                                                float* __restrict__ y, int batch) {
    extern __shared__ __align__(16) uint8_t smem[];
    float* xs = (float*)smem;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t kp = (k_cols + 255) / 256 * 256;
    for (int b = 0; b < batch; ++b)
        for (int64_t c = threadIdx.x; c < kp; c += blockDim.x)
            xs[(int64_t)b * kp + c] = c < k_cols ? __uint_as_float((uint32_t)x[(int64_t)b * k_cols + c] << 16) : 0.f;
    __syncthreads();
    const bool vec = (k_cols % 8) == 0;
    const int64_t groups = (n_rows + kRowsPerWarp - 1) / kRowsPerWarp;
    const int64_t gw = (int64_t)blockIdx.x * kWarps + warp, nw = (int64_t)gridDim.x * kWarps;
    for (int64_t g = gw; g < groups; g += nw) {
        const int64_t r0 = g * kRowsPerWarp;
        float acc[kRowsPerWarp][B];
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
            for (int b = 0; b < B; ++b) acc[r][b] = 0.f;
        for (int64_t c = 8 * lane; c < k_cols; c += 256) {
            uint4 v[kRowsPerWarp];
#pragma unroll
            for (int r = 0; r < kRowsPerWarp; ++r) {
                v[r] = make_uint4(0, 0, 0, 0);
                if (r0 + r < n_rows) {
                    const uint16_t* src = w + (r0 + r) * k_cols + c;
                    if (vec) {
                        v[r] = __ldg((const uint4*)src);
                    } else {
                        uint16_t h[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j) h[j] = c + j < k_cols ? src[j] : 0;
                        v[r] = make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16), h[6] | (h[7] << 16));
                    }
                }
            }
#pragma unroll
            for (int b = 0; b < B; ++b) {
                if (b >= batch) break;
                const float4 xa = *(const float4*)(xs + (int64_t)b * kp + c);
                const float4 xb = *(const float4*)(xs + (int64_t)b * kp + c + 4);
#pragma unroll
                for (int r = 0; r < kRowsPerWarp; ++r) {
                    const uint32_t q[4] = {v[r].x, v[r].y, v[r].z, v[r].w};
                    float s = acc[r][b];
                    s = fmaf(__uint_as_float(q[0] << 16), xa.x, s);
                    s = fmaf(__uint_as_float(q[0] & 0xFFFF0000u), xa.y, s);
                    s = fmaf(__uint_as_float(q[1] << 16), xa.z, s);
                    s = fmaf(__uint_as_float(q[1] & 0xFFFF0000u), xa.w, s);
                    s = fmaf(__uint_as_float(q[2] << 16), xb.x, s);
                    s = fmaf(__uint_as_float(q[2] & 0xFFFF0000u), xb.y, s);
                    s = fmaf(__uint_as_float(q[3] << 16), xb.z, s);
                    s = fmaf(__uint_as_float(q[3] & 0xFFFF0000u), xb.w, s);
                    acc[r][b] = s;
                }
            }
        }
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
            for (int b = 0; b < B; ++b) {
                if (b >= batch) break;
                const float v = warp_sum(acc[r][b]);
                if (lane == 0 && r0 + r < n_rows) y[(int64_t)b * n_rows + r0 + r] = v;
            }
    }
}

/* ============================================================ host helpers */
struct DeviceInfo {
    int sms = 0;
    size_t smem_optin = 0;
    int* status = nullptr;
};

std::mutex g_mu;
std::vector<DeviceInfo> g_dev;

int device_info(int dev, DeviceInfo** out) {
    std::lock_guard<std::mutex> lk(g_mu);
    if ((int)g_dev.size() <= dev) g_dev.resize(dev + 1);
    DeviceInfo& d = g_dev[dev];
    if (!d.sms) {
        cudaDeviceProp p;
        if (cudaGetDeviceProperties(&p, dev) != cudaSuccess) return EC_ERR_CUDA;
        d.sms = p.multiProcessorCount;
        d.smem_optin = p.sharedMemPerBlockOptin;
        int prev = 0;
        cudaGetDevice(&prev);
        cudaSetDevice(dev);
        const cudaError_t e = cudaMalloc((void**)&d.status, sizeof(int));
        if (e == cudaSuccess) cudaMemset(d.status, 0, sizeof(int));
        cudaSetDevice(prev);
        if (e != cudaSuccess) {
            d.sms = 0;
            return EC_ERR_OOM;
        }
    }
    *out = &d;
    return EC_OK;
}

int current_device(int* dev) { return cudaGetDevice(dev) == cudaSuccess ? EC_OK : EC_ERR_CUDA; }

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

/* Raise a kernel's dynamic shared-memory limit once per (device, kernel); later
 * calls that need no more than the recorded value skip the runtime call. */
template <class K>
int set_smem(K kernel, size_t bytes) {
    struct Entry {
        int dev;
        const void* fn;
        size_t bytes;
    };
    static std::mutex mu;
    static std::vector<Entry> done;
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lk(mu);
    for (Entry& e : done)
        if (e.dev == dev && e.fn == (const void*)kernel) {
            if (bytes <= e.bytes) return EC_OK;
            if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) != cudaSuccess)
                return EC_ERR_CUDA;
            e.bytes = bytes;
            return EC_OK;
        }
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) != cudaSuccess)
        return EC_ERR_CUDA;
    done.push_back({dev, (const void*)kernel, bytes});
    return EC_OK;
}

int launch_result() {
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? EC_OK : EC_ERR_CUDA;
}

/* Programmatic dependent launch: a kernel may start its prologue (tables into
 * shared memory) while the previous kernel in the stream drains; it waits for
 * that kernel (griddepcontrol.wait) before it reads x or writes outputs.
 * EC_NO_PDL=1 in the environment turns it off. */
bool use_pdl() {
    static const bool on = [] {
        const char* e = std::getenv("EC_NO_PDL");
        return !(e && e[0] == '1');
    }();
    return on;
}

template <class... KArgs, class... Args>
int launch_ex(void (*kernel)(KArgs...), int grid, int block, size_t smem, cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = use_pdl() ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, args...) == cudaSuccess ? EC_OK : EC_ERR_CUDA;
}

HuffMat huff_desc(const ec_matrix* W) {
    HuffMat m{};
    const ec_blob_header& h = W->hdr;
    m.records = W->d_blob + h.records_off;
    m.tile_off = (const uint32_t*)(W->d_blob + h.tile_off_off);
    m.table = (const uint32_t*)(W->d_blob + h.table_off);
    m.table_words = h.table_words;
    m.n_rows = h.n_rows;
    m.k_cols = h.k_cols;
    m.k_pad = h.k_pad;
    m.n_tiles = h.n_tiles;
    m.records_bytes = h.blob_bytes - h.records_off;
    m.steps = h.steps;
    const int64_t T = 32 * (int64_t)h.steps;
    m.atomic_y = (h.k_pad > 0 && T % h.k_pad == 0) ? 0 : 1;
    return m;
}

RansMat rans_desc(const ec_matrix* W) {
    RansMat m{};
    const ec_blob_header& h = W->hdr;
    m.records = W->d_blob + h.records_off;
    m.tile_off = (const uint32_t*)(W->d_blob + h.tile_off_off);
    m.table = (const uint32_t*)(W->d_blob + h.table_off);
    m.scales = (const uint16_t*)(W->d_blob + h.scales_off);
    m.n_rows = h.n_rows;
    m.k_cols = h.k_cols;
    m.k_pad = h.k_pad;
    m.n_tiles = h.n_tiles;
    m.records_bytes = h.blob_bytes - h.records_off;
    m.steps = h.steps;
    m.prob_bits = h.prob_bits;
    const int64_t T = 32 * (int64_t)h.steps;
    m.atomic_y = (h.k_pad > 0 && T % h.k_pad == 0) ? 0 : 1;
    m.words_cap = (h.max_words + 7) / 8 * 8;
    return m;
}

int check_matrix(const ec_matrix* W, int dev) {
    if (!W || !W->d_blob || W->hdr.magic != EC_BLOB_MAGIC || W->hdr.version != EC_BLOB_VERSION) return EC_ERR_INVALID_ARG;
    if (W->device != dev) return EC_ERR_INVALID_ARG;
    return EC_OK;
}

/* Largest number of warps' worth of per-warp buffers that fits next to `fixed`. */
int grid_for(const DeviceInfo& d, int64_t work_items, int ctas_per_sm) {
    const int64_t full = (int64_t)d.sms * ctas_per_sm;
    const int64_t need = (work_items + kWarps - 1) / kWarps;
    return (int)std::max<int64_t>(1, std::min(full, need));
}

template <int B>
int launch_huff_gemv_b(const HuffGemvArgs& a, size_t smem, int grid, int block, cudaStream_t s) {
    if (set_smem(huff_gemv_kernel<B>, smem) != EC_OK) return EC_ERR_CUDA;
    return launch_ex(huff_gemv_kernel<B>, grid, block, smem, s, a);
}

int launch_huff_gemv(const HuffGemvArgs& a, size_t smem, int grid, int block, cudaStream_t s) {
    if (a.batch <= 1) return launch_huff_gemv_b<1>(a, smem, grid, block, s);
    if (a.batch <= 2) return launch_huff_gemv_b<2>(a, smem, grid, block, s);
    if (a.batch <= 4) return launch_huff_gemv_b<4>(a, smem, grid, block, s);
    if (a.batch <= 8) return launch_huff_gemv_b<8>(a, smem, grid, block, s);
    return launch_huff_gemv_b<16>(a, smem, grid, block, s);
}

template <bool G, int B>
int launch_rans_b(const RansArgs& a, size_t smem, int grid, cudaStream_t s) {
    if (set_smem(rans_kernel<G, B>, smem) != EC_OK) return EC_ERR_CUDA;
    rans_kernel<G, B><<<grid, kWarps * 32, smem, s>>>(a);
    return launch_result();
}

int launch_rans(bool gemv, const RansArgs& a, size_t smem, int grid, cudaStream_t s) {
    if (!gemv) return launch_rans_b<false, 1>(a, smem, grid, s);
    if (a.batch <= 1) return launch_rans_b<true, 1>(a, smem, grid, s);
    if (a.batch <= 2) return launch_rans_b<true, 2>(a, smem, grid, s);
    if (a.batch <= 4) return launch_rans_b<true, 4>(a, smem, grid, s);
    if (a.batch <= 8) return launch_rans_b<true, 8>(a, smem, grid, s);
    return launch_rans_b<true, 16>(a, smem, grid, s);
}

/* Batch rows whose copy of x (elem bytes per value) fits in `budget` bytes of shared memory. */
int rows_per_pass(int64_t k_pad, int batch, size_t budget, int elem = 4) {
    if (k_pad == 0) return batch;
    const int64_t per = elem * k_pad;
    return (int)std::max<int64_t>(0, std::min<int64_t>(batch, (int64_t)budget / per));
}

/* ----------------------------------------------------------- Huffman GEMV */
int huff_gemv(const ec_matrix* const* Ws, int count, const uint16_t* x, float* const* ys, int batch,
              cudaStream_t s, int dev, DeviceInfo* d) {
    int64_t total = 0;
    int code_bytes = 16;
    HuffGemvArgs a{};
    a.count = count;
    const int64_t K = Ws[0]->hdr.k_cols, kp = Ws[0]->hdr.k_pad;
    for (int k = 0; k < count; ++k) {
        const ec_matrix* W = Ws[k];
        a.m[k] = huff_desc(W);
        a.m[k].tile_begin = total;
        total += W->hdr.n_tiles;
        code_bytes = std::max(code_bytes, (int)W->hdr.max_code_bytes);
        if (a.m[k].atomic_y || W->hdr.n_tiles == 0) {
            if (cudaMemsetAsync(ys[k], 0, sizeof(float) * (size_t)batch * (size_t)W->hdr.n_rows, s) != cudaSuccess)
                return EC_ERR_CUDA;
        }
    }
    code_bytes = (code_bytes + 15) & ~15;
    a.total_tiles = total;
    a.status = d->status;
    a.code_bytes = code_bytes;
    if (total == 0) return EC_OK;
    /* warps per CTA: as many as fit next to the tables and one batch row of x (>= 4) */
    const size_t tables = (size_t)count * kMultiBytes, per_warp = huff_warp_bytes(code_bytes);
    const size_t xrow = xs_row_bytes((uint32_t)kp);
    if (tables + xrow + 4 * per_warp > d->smem_optin) return EC_ERR_UNSUPPORTED;
    const int warps = (int)std::min<size_t>(kHW, (d->smem_optin - tables - xrow) / per_warp);
    const size_t fixed = tables + (size_t)warps * per_warp;
    const int per_pass = (int)std::min<size_t>(batch, (d->smem_optin - fixed) / xrow);
    if (per_pass < 1) return EC_ERR_UNSUPPORTED;
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(d->sms, (total + warps - 1) / warps));
    for (int b0 = 0; b0 < batch; b0 += per_pass) {
        const int nb = std::min(per_pass, batch - b0);
        a.batch = nb;
        a.x = x + (int64_t)b0 * K;
        for (int k = 0; k < count; ++k) a.m[k].y = ys[k] + (int64_t)b0 * Ws[k]->hdr.n_rows;
        const size_t smem = fixed + xrow * nb;
        const int rc = launch_huff_gemv(a, smem, grid, warps * 32, s);
        if (rc != EC_OK) return rc;
    }
    return EC_OK;
}

int rans_run(const ec_matrix* W, const uint16_t* x, float* y, uint16_t* out, int batch, cudaStream_t s,
             DeviceInfo* d) {
    RansArgs a{};
    a.m = rans_desc(W);
    a.m.y = y;
    a.m.out = out;
    a.status = d->status;
    const bool gemv = y != nullptr;
    if (gemv && (a.m.atomic_y || W->hdr.n_tiles == 0)) {
        if (cudaMemsetAsync(y, 0, sizeof(float) * (size_t)batch * (size_t)W->hdr.n_rows, s) != cudaSuccess)
            return EC_ERR_CUDA;
    }
    if (W->hdr.n_tiles == 0) return EC_OK;
    const size_t fixed = ((size_t)4 << a.m.prob_bits) + (size_t)kWarps * 2 * a.m.words_cap;
    if (fixed > d->smem_optin) return EC_ERR_UNSUPPORTED;
    const int64_t kp = W->hdr.k_pad, K = W->hdr.k_cols;
    const int per_pass = gemv ? rows_per_pass(kp, batch, d->smem_optin - fixed) : 1;
    if (per_pass < 1) return EC_ERR_UNSUPPORTED;
    const int passes = gemv ? batch : 1;
    for (int b0 = 0; b0 < passes; b0 += per_pass) {
        const int nb = gemv ? std::min(per_pass, batch - b0) : 0;
        a.batch = nb;
        a.x = gemv ? x + (int64_t)b0 * K : nullptr;
        if (gemv) a.m.y = y + (int64_t)b0 * W->hdr.n_rows;
        const size_t smem = fixed + (size_t)4 * nb * kp;
        const int ctas = std::max(1, (int)(d->smem_optin / (smem + 1024)));
        const int grid = grid_for(*d, W->hdr.n_tiles, std::min(ctas, 2));
        const int rc = launch_rans(gemv, a, smem, grid, s);
        if (rc != EC_OK) return rc;
    }
    return EC_OK;
}

/* ====================================================== allocation-free GEMV */
/* Scratch for ec_gemv_static: one file-scope device array that every GPU loading
 * this library holds until exit.  Word 0 is the status word of those calls; the
 * partial row sums start after a 256-byte header. */
constexpr size_t kStaticScratchBytes = size_t(4) << 20; /* 4 MiB */
constexpr int64_t kStaticHeaderFloats = 64;
constexpr int64_t kStaticPartFloats = (int64_t)(kStaticScratchBytes / sizeof(float)) - kStaticHeaderFloats;
static __device__ __align__(256) float g_ec_static_scratch[kStaticScratchBytes / sizeof(float)];

/* y[b, r] = sum of the row's partial sums, one per tile that covers row r, added in
 * tile order (so the result is the same on every call). */
__global__ void part_reduce_kernel(const float* __restrict__ part, int slots, int64_t n_rows, int64_t k_pad, int64_t T,
                                   int batch, float* __restrict__ y) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (int64_t)batch * n_rows) return;
    const int64_t r = i % n_rows;
    const int64_t first = (r * k_pad) / T, last = ((r + 1) * k_pad - 1) / T;
    const float* src = part + i * slots;
    float s = 0.f;
    for (int64_t k = 0; k <= last - first && k < slots; ++k) s += src[k];
    y[i] = s;
}

/* Per-device set-up of the allocation-free path, in a fixed table (no allocation):
 * SM count, shared-memory limit and the device address of the scratch array. */
struct StaticDevice {
    int ready;
    int sms;
    size_t smem_optin;
    float* scratch;
};
constexpr int kMaxStaticDevices = 64;
StaticDevice g_static_dev[kMaxStaticDevices];
std::mutex g_static_mu;

int static_device(int dev, StaticDevice** out) {
    if (dev < 0 || dev >= kMaxStaticDevices) return EC_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_static_mu);
    StaticDevice& s = g_static_dev[dev];
    if (!s.ready) {
        int sms = 0, optin = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
            return EC_ERR_CUDA;
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_ec_static_scratch) != cudaSuccess || !p) return EC_ERR_CUDA;
        s.sms = sms;
        s.smem_optin = (size_t)optin;
        s.scratch = (float*)p;
        s.ready = 1;
    }
    *out = &s;
    return EC_OK;
}

template <int B>
int launch_huff_gemv_part_b(const HuffGemvArgs& a, size_t smem, int grid, int block, cudaStream_t s) {
    if (cudaFuncSetAttribute(huff_gemv_kernel<B, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return EC_ERR_CUDA;
    return launch_ex(huff_gemv_kernel<B, true>, grid, block, smem, s, a);
}

int launch_huff_gemv_part(const HuffGemvArgs& a, size_t smem, int grid, int block, cudaStream_t s) {
    if (a.batch <= 1) return launch_huff_gemv_part_b<1>(a, smem, grid, block, s);
    if (a.batch <= 2) return launch_huff_gemv_part_b<2>(a, smem, grid, block, s);
    if (a.batch <= 4) return launch_huff_gemv_part_b<4>(a, smem, grid, block, s);
    if (a.batch <= 8) return launch_huff_gemv_part_b<8>(a, smem, grid, block, s);
    return launch_huff_gemv_part_b<16>(a, smem, grid, block, s);
}

}  // namespace

/* ================================================================ C ABI */
extern "C" int ec_gemv_group(const ec_matrix* const* Ws, int count, const uint16_t* x, float* const* ys, int batch,
                             cudaStream_t stream) {
    if (!Ws || !ys || count < 1 || count > EC_MAX_GROUP) return EC_ERR_INVALID_ARG;
    if (batch < 1 || batch > EC_MAX_BATCH) return batch < 1 ? EC_ERR_INVALID_ARG : EC_ERR_UNSUPPORTED;
    for (int k = 0; k < count; ++k)
        if (!Ws[k] || !Ws[k]->d_blob) return EC_ERR_INVALID_ARG; /* null or host-only matrix */
    int dev = 0;
    if (current_device(&dev) != EC_OK) return EC_ERR_CUDA;
    DeviceInfo* d = nullptr;
    int rc = device_info(dev, &d);
    if (rc != EC_OK) return rc;
    for (int k = 0; k < count; ++k) {
        if ((rc = check_matrix(Ws[k], dev)) != EC_OK) return rc;
        if (Ws[k]->kind != Ws[0]->kind || Ws[k]->hdr.k_cols != Ws[0]->hdr.k_cols) return EC_ERR_SHAPE;
        if (!ys[k] || !aligned16(ys[k])) return EC_ERR_INVALID_ARG;
    }
    if (Ws[0]->hdr.k_cols > 0 && (!x || !aligned16(x))) return EC_ERR_INVALID_ARG;
    if (Ws[0]->kind == EC_KIND_HUFFMAN_BF16) return huff_gemv(Ws, count, x, ys, batch, stream, dev, d);
    for (int k = 0; k < count; ++k)
        if ((rc = rans_run(Ws[k], x, ys[k], nullptr, batch, stream, d)) != EC_OK) return rc;
    return EC_OK;
}

extern "C" int ec_gemv(const ec_matrix* W, const uint16_t* x, float* y, int batch, cudaStream_t stream) {
    return ec_gemv_group(&W, 1, x, &y, batch, stream);
}

extern "C" int ec_decode_batch(const ec_matrix* const* Ws, uint16_t* const* outs, int count, cudaStream_t stream) {
    if (!Ws || !outs || count < 1 || count > kMaxDecodeBatch) return EC_ERR_INVALID_ARG;
    for (int k = 0; k < count; ++k)
        if (!Ws[k] || !Ws[k]->d_blob) return EC_ERR_INVALID_ARG;
    int dev = 0;
    if (current_device(&dev) != EC_OK) return EC_ERR_CUDA;
    DeviceInfo* d = nullptr;
    int rc = device_info(dev, &d);
    if (rc != EC_OK) return rc;
    HuffDecodeArgs a{};
    int64_t total = 0;
    int code_bytes = 16;
    for (int k = 0; k < count; ++k) {
        if ((rc = check_matrix(Ws[k], dev)) != EC_OK) return rc;
        const int64_t n = Ws[k]->hdr.n_rows * Ws[k]->hdr.k_cols;
        if (n > 0 && (!outs[k] || !aligned16(outs[k]))) return EC_ERR_INVALID_ARG;
        if (Ws[k]->kind == EC_KIND_RANS_INT4) {
            if ((rc = rans_run(Ws[k], nullptr, nullptr, outs[k], 1, stream, d)) != EC_OK) return rc;
            continue;
        }
        HuffMat m = huff_desc(Ws[k]);
        m.out = outs[k];
        m.tile_begin = total;
        total += Ws[k]->hdr.n_tiles;
        code_bytes = std::max(code_bytes, (int)Ws[k]->hdr.max_code_bytes);
        a.m[a.count++] = m;
    }
    if (a.count == 0 || total == 0) return EC_OK;
    code_bytes = (code_bytes + 15) & ~15;
    a.total_tiles = total;
    a.status = d->status;
    a.code_bytes = code_bytes;
    const size_t per_warp = decode_warp_bytes(code_bytes);
    if (kMultiBytes + 4 * per_warp > d->smem_optin) return EC_ERR_UNSUPPORTED;
    const int warps = (int)std::min<size_t>(kHW, (d->smem_optin - kMultiBytes) / per_warp);
    const size_t smem = kMultiBytes + (size_t)warps * per_warp;
    if (set_smem(huff_decode_kernel, smem) != EC_OK) return EC_ERR_CUDA;
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(d->sms, (total + warps - 1) / warps));
    return launch_ex(huff_decode_kernel, grid, warps * 32, smem, stream, a);
}

extern "C" int ec_decode(const ec_matrix* W, uint16_t* out, cudaStream_t stream) {
    return ec_decode_batch(&W, &out, 1, stream);
}

extern "C" int ec_bf16_gemv(const uint16_t* w, int64_t n_rows, int64_t k_cols, const uint16_t* x, float* y, int batch,
                            cudaStream_t stream) {
    if (n_rows < 0 || k_cols < 0) return EC_ERR_SHAPE;
    if (batch < 1) return EC_ERR_INVALID_ARG;
    if (batch > EC_MAX_BATCH) return EC_ERR_UNSUPPORTED;
    if (n_rows == 0) return EC_OK;
    if (!y || !aligned16(y) || (k_cols > 0 && (!w || !x || !aligned16(w) || !aligned16(x)))) return EC_ERR_INVALID_ARG;
    int dev = 0;
    if (current_device(&dev) != EC_OK) return EC_ERR_CUDA;
    DeviceInfo* d = nullptr;
    int rc = device_info(dev, &d);
    if (rc != EC_OK) return rc;
    const int64_t kp = (k_cols + 255) / 256 * 256;
    const int per_pass = rows_per_pass(kp, batch, d->smem_optin);
    if (per_pass < 1) return EC_ERR_UNSUPPORTED;
    const int64_t groups = (n_rows + kRowsPerWarp - 1) / kRowsPerWarp;
    for (int b0 = 0; b0 < batch; b0 += per_pass) {
        const int nb = std::min(per_pass, batch - b0);
        const size_t smem = std::max<size_t>((size_t)4 * nb * kp, 16);
        const int ctas = std::max(1, std::min(4, (int)(d->smem_optin / (smem + 1024))));
        const int grid = grid_for(*d, groups, ctas);
        const uint16_t* xb = x + (int64_t)b0 * k_cols;
        float* yb = y + (int64_t)b0 * n_rows;
#define EC_BF16_LAUNCH(BB)                                                                      \
    do {                                                                                        \
        if (set_smem(bf16_gemv_kernel<BB>, smem) != EC_OK) return EC_ERR_CUDA;                  \
        bf16_gemv_kernel<BB><<<grid, kWarps * 32, smem, stream>>>(w, n_rows, k_cols, xb, yb, nb); \
    } while (0)
        if (nb <= 1) EC_BF16_LAUNCH(1);
        else if (nb <= 2) EC_BF16_LAUNCH(2);
        else if (nb <= 4) EC_BF16_LAUNCH(4);
        else if (nb <= 8) EC_BF16_LAUNCH(8);
        else EC_BF16_LAUNCH(16);
#undef EC_BF16_LAUNCH
        const int rc = launch_result();
        if (rc != EC_OK) return rc;
    }
    return EC_OK;
}

extern "C" int ec_status(cudaStream_t stream) {
    if (cudaStreamSynchronize(stream) != cudaSuccess) return EC_ERR_CUDA;
    int dev = 0;
    if (current_device(&dev) != EC_OK) return EC_ERR_CUDA;
    DeviceInfo* d = nullptr;
    int rc = device_info(dev, &d);
    if (rc != EC_OK) return rc;
    int v = 0;
    if (cudaMemcpy(&v, d->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return EC_ERR_CUDA;
    if (v && cudaMemset(d->status, 0, sizeof(int)) != cudaSuccess) return EC_ERR_CUDA;
    return v ? EC_ERR_CORRUPT : EC_OK;
}

/* Allocation-free GEMV (declared in ec.h, where its contract is described). */
extern "C" int ec_gemv_static(const ec_matrix* W, const uint16_t* x, float* y, int batch, cudaStream_t stream) {
    if (!W || !W->d_blob) return EC_ERR_INVALID_ARG;
    if (batch < 1) return EC_ERR_INVALID_ARG;
    if (batch > EC_MAX_BATCH || W->kind != EC_KIND_HUFFMAN_BF16) return EC_ERR_UNSUPPORTED;
    if (!y || !aligned16(y) || (W->hdr.k_cols > 0 && (!x || !aligned16(x)))) return EC_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return EC_ERR_CUDA;
    if (check_matrix(W, dev) != EC_OK) return EC_ERR_INVALID_ARG;
    StaticDevice* d = nullptr;
    int rc = static_device(dev, &d);
    if (rc != EC_OK) return rc;
    const ec_blob_header& h = W->hdr;
    const int64_t T = 32 * (int64_t)h.steps;
    const int64_t slots = (h.k_pad + T - 1) / T + 1;
    if (h.n_rows > 0 && (int64_t)batch * slots > kStaticPartFloats / h.n_rows) return EC_ERR_UNSUPPORTED;
    if (h.n_tiles == 0)
        return cudaMemsetAsync(y, 0, sizeof(float) * (size_t)batch * (size_t)h.n_rows, stream) == cudaSuccess
                   ? EC_OK
                   : EC_ERR_CUDA;
    HuffGemvArgs a{};
    a.m[0] = huff_desc(W);
    a.count = 1;
    a.total_tiles = h.n_tiles;
    a.status = (int*)d->scratch;
    a.code_bytes = ((int)h.max_code_bytes + 15) & ~15;
    a.part = d->scratch + kStaticHeaderFloats;
    a.part_slots = (int)slots;
    if (a.code_bytes < 16) a.code_bytes = 16;
    if (cudaMemsetAsync(d->scratch, 0, sizeof(int), stream) != cudaSuccess) return EC_ERR_CUDA;
    const size_t tables = kMultiBytes, per_warp = huff_warp_bytes(a.code_bytes);
    const size_t xrow = xs_row_bytes((uint32_t)h.k_pad);
    if (tables + xrow + 4 * per_warp > d->smem_optin) return EC_ERR_UNSUPPORTED;
    const int warps = (int)std::min<size_t>(kHW, (d->smem_optin - tables - xrow) / per_warp);
    const size_t fixed = tables + (size_t)warps * per_warp;
    const int per_pass = (int)std::min<size_t>(batch, (d->smem_optin - fixed) / xrow);
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(d->sms, (h.n_tiles + warps - 1) / warps));
    for (int b0 = 0; b0 < batch; b0 += per_pass) {
        const int nb = std::min(per_pass, batch - b0);
        a.batch = nb;
        a.x = x + (int64_t)b0 * h.k_cols;
        if ((rc = launch_huff_gemv_part(a, fixed + xrow * nb, grid, warps * 32, stream)) != EC_OK) return rc;
        const int64_t n = (int64_t)nb * h.n_rows;
        part_reduce_kernel<<<(unsigned)((n + 255) / 256), 256, 0, stream>>>(a.part, a.part_slots, h.n_rows, h.k_pad,
                                                                           T, nb, y + (int64_t)b0 * h.n_rows);
        if ((rc = launch_result()) != EC_OK) return rc;
    }
    return EC_OK;
}
