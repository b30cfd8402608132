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
#include <cstring>
#include <mutex>
#include <vector>

#include "ec_internal.h"

namespace {

constexpr int kWarps = 8;          /* warps per CTA */
constexpr int kChunk = 32;         /* steps decoded before each multiply-accumulate pass */
constexpr int kStage = (kChunk + 4) * 32 * 2; /* per-warp exponent stage (bytes), with slack */
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

/* Sub-table walk for codewords longer than the level-1 window. */
__device__ __noinline__ uint32_t walk_subtables(uint32_t ent, uint32_t win, const uint32_t* __restrict__ table,
                                                int64_t table_words, int* status) {
#pragma unroll 1
    for (int lvl = 0; lvl < 3 && (ent & EC_ENT_PTR); ++lvl) {
        const int used = (int)((ent >> 16) & 31);
        const int64_t at = (int64_t(1) << EC_L1_BITS) + (int64_t)(ent & 0xFFFFu) * 256 + ((win << used) >> 24);
        if (used > 24 || at >= table_words) {
            ent = EC_ENT_BAD;
            break;
        }
        ent = __ldg(table + at);
    }
    if (ent & (EC_ENT_PTR | EC_ENT_BAD)) {
        flag_corrupt(status);
        ent = 1u << 16; /* length 1, exponent 0: keeps the lane moving */
    }
    return ent;
}

/* Decode `n` codewords of one lane into stage[i * 32 + lane] (16-bit exponent
 * fields).  (hi, lo) is the 64-bit window, pos the bits already consumed in hi. */
struct LaneDecoder {
    uint32_t hi, lo;
    int pos, widx;
};

__device__ __forceinline__ void lane_init(LaneDecoder& d, const uint32_t* area, int area_words, int start_byte) {
    const int w = start_byte >> 2;
    d.pos = (start_byte & 3) * 8;
    d.hi = w < area_words ? area[w] : 0u;
    d.lo = w + 1 < area_words ? area[w + 1] : 0u;
    d.widx = w + 2;
}

__device__ __forceinline__ void lane_decode(LaneDecoder& d, int n, const uint32_t* __restrict__ l1, const uint32_t* area,
                                            int area_words, uint16_t* stage, int lane,
                                            const uint32_t* __restrict__ table, int64_t table_words, int* status) {
#pragma unroll 4
    for (int i = 0; i < n; ++i) {
        const uint32_t win = __funnelshift_l(d.lo, d.hi, d.pos);
        uint32_t ent = l1[win >> (32 - EC_L1_BITS)];
        if (ent & (EC_ENT_PTR | EC_ENT_BAD)) ent = walk_subtables(ent, win, table, table_words, status);
        stage[i * 32 + lane] = (uint16_t)ent;
        d.pos += (int)((ent >> 16) & 31);
        if (d.pos >= 32) {
            d.hi = d.lo;
            d.lo = d.widx < area_words ? area[d.widx] : 0u;
            d.widx++;
            d.pos -= 32;
        }
    }
}

/* Merge two exponent fields (e0, e1 in the low / high half of e) with raw bytes
 * r0 = byte a, r1 = byte a+1 of r into two BF16 values [w1 | w0]. */
__device__ __forceinline__ uint32_t merge_pair(uint32_t e, uint32_t r, uint32_t sel) {
    const uint32_t dup = __byte_perm(r, 0, sel); /* [r1 r1 r0 r0] */
    return e | (dup & 0x807F807Fu);
}

/* Eight BF16 weights for 8 consecutive positions: stage fields e8, raw bytes r8. */
__device__ __forceinline__ void merge8(const uint4& e8, const uint2& r8, uint32_t (&p)[4]) {
    p[0] = merge_pair(e8.x, r8.x, 0x1100);
    p[1] = merge_pair(e8.y, r8.x, 0x3322);
    p[2] = merge_pair(e8.z, r8.y, 0x1100);
    p[3] = merge_pair(e8.w, r8.y, 0x3322);
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

/* ======================================================== Huffman GEMV kernel */
template <int B>
__global__ void __launch_bounds__(kWarps * 32) huff_gemv_kernel(const __grid_constant__ HuffGemvArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t kp = a.m[0].k_pad;
    const int batch = a.batch;

    /* shared: level-1 tables | x (fp32, [batch, k_pad]) | per warp: code buffer + stage */
    uint32_t* l1s = (uint32_t*)smem;
    float* xs = (float*)(smem + (size_t)a.count * (4u << EC_L1_BITS));
    uint8_t* wbase = (uint8_t*)(xs + (size_t)batch * kp) + (size_t)warp * (a.code_bytes + kStage);
    uint32_t* code = (uint32_t*)wbase;
    uint16_t* stage = (uint16_t*)(wbase + a.code_bytes);

    for (int k = 0; k < a.count; ++k)
        for (int i = threadIdx.x; i < (1 << EC_L1_BITS); i += blockDim.x) l1s[(k << EC_L1_BITS) + i] = __ldg(a.m[k].table + i);
    const int64_t K = a.m[0].k_cols;
    for (int b = 0; b < batch; ++b)
        for (int64_t c = threadIdx.x; c < kp; c += blockDim.x) {
            float v = 0.f;
            if (c < K) v = __uint_as_float((uint32_t)a.x[(int64_t)b * K + c] << 16);
            xs[(int64_t)b * kp + c] = v;
        }
    __syncthreads();

    const int64_t gw = (int64_t)blockIdx.x * kWarps + warp, nw = (int64_t)gridDim.x * kWarps;
    for (int64_t g = gw; g < a.total_tiles; g += nw) {
        const int mi = owner(a, g);
        const HuffMat& M = a.m[mi];
        const int64_t t = g - M.tile_begin;
        const int64_t T = 32 * (int64_t)M.steps;
        const int64_t base = t * T;
        const int64_t n_t = min(T, M.n_rows * kp - base);
        const int S = (int)(n_t / 32);
        int64_t rec_bytes = 0;
        const uint8_t* rec = M.records + record_span(M.tile_off, t, M.records_bytes, &rec_bytes, a.status, lane);
        const int raw_bytes = (int)((n_t + 15) & ~15);
        if (rec_bytes < 64 + raw_bytes) { /* corrupt offsets: skip the tile */
            if (lane == 0) flag_corrupt(a.status);
            continue;
        }
        int area_bytes = (int)(rec_bytes - 64 - raw_bytes);
        if (area_bytes < 0 || area_bytes > a.code_bytes) {
            if (lane == 0) flag_corrupt(a.status);
            area_bytes = max(0, min(area_bytes, a.code_bytes));
        }
        const int area_words = area_bytes / 4;
        const uint16_t start = __ldg((const uint16_t*)rec + lane);
        const uint8_t* raw = rec + 64;
        warp_copy16(code, rec + 64 + raw_bytes, area_bytes, lane);
        __syncwarp();
        const uint32_t* l1 = l1s + (mi << EC_L1_BITS);

        LaneDecoder dec;
        lane_init(dec, code, area_words, start);
        int64_t row = tile_row(t, T, kp, EC_HUFF_ROW_ALIGN);
        int64_t col0 = base - row * kp;
        float acc[B];
#pragma unroll
        for (int b = 0; b < B; ++b) acc[b] = 0.f;

        auto flush = [&](int64_t r) {
#pragma unroll
            for (int b = 0; b < B; ++b) {
                if (b >= batch) break;
                const float v = warp_sum(acc[b]);
                if (lane == 0) {
                    float* dst = M.y + (int64_t)b * M.n_rows + r;
                    if (M.atomic_y) atomicAdd(dst, v);
                    else *dst = v;
                }
                acc[b] = 0.f;
            }
        };

        for (int c0 = 0; c0 < S; c0 += kChunk) {
            const int n = min(kChunk, S - c0);
            const int subs = n / 8;
            uint2 r8[kChunk / 8];
#pragma unroll
            for (int k = 0; k < kChunk / 8; ++k)
                if (k < subs) r8[k] = __ldg((const uint2*)(raw + (int64_t)c0 * 32 + k * 256) + lane);
            lane_decode(dec, n, l1, code, area_words, stage, lane, M.table, M.table_words, a.status);
            __syncwarp();
#pragma unroll
            for (int k = 0; k < kChunk / 8; ++k) {
                if (k >= subs) break;
                if (col0 >= kp) {
                    flush(row);
                    col0 -= kp;
                    ++row;
                }
                const uint4 e8 = *(const uint4*)(stage + k * 256 + 8 * lane);
                uint32_t p[4];
                merge8(e8, r8[k], p);
                float w[8];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    w[2 * j] = __uint_as_float(p[j] << 16);
                    w[2 * j + 1] = __uint_as_float(p[j] & 0xFFFF0000u);
                }
                const int64_t col = col0 + 8 * lane;
#pragma unroll
                for (int b = 0; b < B; ++b) {
                    if (b >= batch) break;
                    const float4 xa = *(const float4*)(xs + (int64_t)b * kp + col);
                    const float4 xb = *(const float4*)(xs + (int64_t)b * kp + col + 4);
                    float s = acc[b];
                    s = fmaf(w[0], xa.x, s);
                    s = fmaf(w[1], xa.y, s);
                    s = fmaf(w[2], xa.z, s);
                    s = fmaf(w[3], xa.w, s);
                    s = fmaf(w[4], xb.x, s);
                    s = fmaf(w[5], xb.y, s);
                    s = fmaf(w[6], xb.z, s);
                    s = fmaf(w[7], xb.w, s);
                    acc[b] = s;
                }
                col0 += 256;
            }
            __syncwarp();
        }
        flush(row);
    }
}

/* ====================================================== Huffman decode kernel */
__global__ void __launch_bounds__(kWarps * 32) huff_decode_kernel(const __grid_constant__ HuffDecodeArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint8_t* wbase = smem + (size_t)warp * (a.code_bytes + kStage + (4u << EC_L1_BITS));
    uint32_t* l1w = (uint32_t*)wbase; /* per-warp copy: matrices differ between warps */
    uint32_t* code = (uint32_t*)(wbase + (4u << EC_L1_BITS));
    uint16_t* stage = (uint16_t*)(wbase + (4u << EC_L1_BITS) + a.code_bytes);
    int loaded = -1;

    const int64_t gw = (int64_t)blockIdx.x * kWarps + warp, nw = (int64_t)gridDim.x * kWarps;
    for (int64_t g = gw; g < a.total_tiles; g += nw) {
        const int mi = owner(a, g);
        const HuffMat& M = a.m[mi];
        if (mi != loaded) {
            __syncwarp();
            for (int i = lane; i < (1 << EC_L1_BITS); i += 32) l1w[i] = __ldg(M.table + i);
            loaded = mi;
            __syncwarp();
        }
        const int64_t kp = M.k_pad, K = M.k_cols;
        const int64_t t = g - M.tile_begin;
        const int64_t T = 32 * (int64_t)M.steps;
        const int64_t base = t * T;
        const int64_t n_t = min(T, M.n_rows * kp - base);
        const int S = (int)(n_t / 32);
        int64_t rec_bytes = 0;
        const uint8_t* rec = M.records + record_span(M.tile_off, t, M.records_bytes, &rec_bytes, a.status, lane);
        const int raw_bytes = (int)((n_t + 15) & ~15);
        if (rec_bytes < 64 + raw_bytes) { /* corrupt offsets: skip the tile */
            if (lane == 0) flag_corrupt(a.status);
            continue;
        }
        int area_bytes = (int)(rec_bytes - 64 - raw_bytes);
        if (area_bytes < 0 || area_bytes > a.code_bytes) {
            if (lane == 0) flag_corrupt(a.status);
            area_bytes = max(0, min(area_bytes, a.code_bytes));
        }
        const int area_words = area_bytes / 4;
        const uint16_t start = __ldg((const uint16_t*)rec + lane);
        const uint8_t* raw = rec + 64;
        warp_copy16(code, rec + 64 + raw_bytes, area_bytes, lane);
        __syncwarp();

        LaneDecoder dec;
        lane_init(dec, code, area_words, start);
        int64_t row = tile_row(t, T, kp, EC_HUFF_ROW_ALIGN);
        int64_t col0 = base - row * kp;
        const bool vec = (K % 8) == 0;
        for (int c0 = 0; c0 < S; c0 += kChunk) {
            const int n = min(kChunk, S - c0);
            const int subs = n / 8;
            uint2 r8[kChunk / 8];
#pragma unroll
            for (int k = 0; k < kChunk / 8; ++k)
                if (k < subs) r8[k] = __ldg((const uint2*)(raw + (int64_t)c0 * 32 + k * 256) + lane);
            lane_decode(dec, n, l1w, code, area_words, stage, lane, M.table, M.table_words, a.status);
            __syncwarp();
#pragma unroll
            for (int k = 0; k < kChunk / 8; ++k) {
                if (k >= subs) break;
                if (col0 >= kp) {
                    col0 -= kp;
                    ++row;
                }
                const uint4 e8 = *(const uint4*)(stage + k * 256 + 8 * lane);
                uint32_t p[4];
                merge8(e8, r8[k], p);
                const int64_t col = col0 + 8 * lane;
                uint16_t* dst = M.out + row * K + col;
                if (vec) {
                    if (col < K) *(uint4*)dst = make_uint4(p[0], p[1], p[2], p[3]);
                } else {
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        if (col + j < K) dst[j] = (uint16_t)(p[j >> 1] >> (16 * (j & 1)));
                }
                col0 += 256;
            }
            __syncwarp();
        }
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
int launch_huff_gemv_b(const HuffGemvArgs& a, size_t smem, int grid, cudaStream_t s) {
    if (set_smem(huff_gemv_kernel<B>, smem) != EC_OK) return EC_ERR_CUDA;
    huff_gemv_kernel<B><<<grid, kWarps * 32, smem, s>>>(a);
    return launch_result();
}

int launch_huff_gemv(const HuffGemvArgs& a, size_t smem, int grid, cudaStream_t s) {
    if (a.batch <= 1) return launch_huff_gemv_b<1>(a, smem, grid, s);
    if (a.batch <= 2) return launch_huff_gemv_b<2>(a, smem, grid, s);
    if (a.batch <= 4) return launch_huff_gemv_b<4>(a, smem, grid, s);
    if (a.batch <= 8) return launch_huff_gemv_b<8>(a, smem, grid, s);
    return launch_huff_gemv_b<16>(a, smem, grid, s);
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

/* Batch rows whose FP32 copy of x fits in `budget` bytes of shared memory. */
int rows_per_pass(int64_t k_pad, int batch, size_t budget) {
    if (k_pad == 0) return batch;
    const int64_t per = 4 * k_pad;
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
    const size_t fixed = (size_t)count * (4u << EC_L1_BITS) + (size_t)kWarps * (code_bytes + kStage);
    if (fixed > d->smem_optin) return EC_ERR_UNSUPPORTED;
    int per_pass = rows_per_pass(kp, batch, d->smem_optin - fixed);
    if (per_pass < 1) return EC_ERR_UNSUPPORTED;
    for (int b0 = 0; b0 < batch; b0 += per_pass) {
        const int nb = std::min(per_pass, batch - b0);
        a.batch = nb;
        a.x = x + (int64_t)b0 * K;
        for (int k = 0; k < count; ++k) a.m[k].y = ys[k] + (int64_t)b0 * Ws[k]->hdr.n_rows;
        const size_t smem = fixed + (size_t)4 * nb * kp;
        const int ctas = std::max(1, (int)(d->smem_optin / (smem + 1024)));
        const int grid = grid_for(*d, total, std::min(ctas, 2));
        const int rc = launch_huff_gemv(a, smem, grid, s);
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
    const size_t smem = (size_t)kWarps * (code_bytes + kStage + (4u << EC_L1_BITS));
    if (smem > d->smem_optin) return EC_ERR_UNSUPPORTED;
    if (set_smem(huff_decode_kernel, smem) != EC_OK) return EC_ERR_CUDA;
    const int ctas = std::max(1, std::min(2, (int)(d->smem_optin / (smem + 1024))));
    huff_decode_kernel<<<grid_for(*d, total, ctas), kWarps * 32, smem, stream>>>(a);
    return launch_result();
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
