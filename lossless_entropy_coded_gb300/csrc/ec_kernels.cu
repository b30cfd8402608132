/*
 * ec_kernels.cu -- sm_103a kernels and the device-side entry points of the C ABI
 * (ec_decode, ec_decode_batch, ec_gemv, ec_gemv_group, ec_gemv_path,
 * ec_gemv_static, ec_bf16_gemv, ec_status).
 *
 * Huffman path (DFloat11, "70% Size, 100% Accuracy", Algorithm 1, re-cut for the
 * fused product of MINE section 4 "Fused mvm"): one warp owns one tile of
 * 32 * steps weights; lane l decodes its own codeword sequence (8 consecutive
 * positions out of every 256: 8 l .. 8 l + 7, 256 + 8 l .. 256 + 8 l + 7, ...)
 * from a byte offset stored in the tile record.  Every lookup of a
 * 12-bit pair table in shared memory yields two exponents already in BF16
 * position; a window whose two codewords do not both fit takes a second lookup,
 * and codewords longer than the window (only when the caller asks for a limit
 * above 12 bits) walk the hierarchical table of DFloat11 Fig. 4 / 14 in global
 * memory.  The decoded pair is merged with the raw sign/mantissa bytes
 *     bf16 = (sign << 15) | (exponent << 7) | mantissa      (Algorithm 1 / Eq. (1))
 * in registers and either stored (decode: one 16-byte store per lane per 8
 * symbols) or multiplied with x in FP32 (GEMV).  Row sums are reduced across the warp with
 * shuffles and written once, or added atomically when a row spans tiles.
 *
 * rANS path (EntroPack, independent rANS tiles): one warp per tile, lane l
 * decodes positions 32 j + l; a lane whose state drops below 2^16 pulls the next
 * 16-bit word, the lanes of one step taking consecutive words in lane order
 * (ballot + popc).  w = code * scale (FP16 scale per 128 weights) is exact in FP32.
 *
 * Robustness: every loop has a fixed trip count; reads of code words, sub-tables
 * and payload words are clamped to the tile / table and inconsistent records or
 * streams set the device status word (EC_ERR_CORRUPT) instead of faulting.
 */
#include <cuda.h> /* CUtensorMap and its encoder's signature (reached through the runtime) */
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <numeric>
#include <vector>

#include "ec_internal.h"

namespace {

constexpr int kWarps = 8;          /* warps per CTA (rANS and BF16 kernels) */
constexpr unsigned kFull = 0xFFFFFFFFu;
constexpr int kMaxDecodeBatch = EC_MAX_DECODE_BATCH;
constexpr int kFmaMaxRows = 16;   /* batch rows per pass of the CUDA-core GEMV kernels */

/* ------------------------------------------------------------ descriptors */
struct HuffMat {
    const uint8_t* records;
    const uint32_t* tile_off;   /* 16-byte units */
    const uint32_t* table;      /* pair table, then the hierarchical sub-tables */
    int64_t table_words;
    int32_t n_sub;              /* hierarchical sub-tables (256 entries each) */
    int32_t fill;               /* the exponent coded in place of a recorded one */
    int32_t sub_smem;           /* their first word in the launch's staged sub-tables, or -1 (global) */
    float* y;                   /* GEMV output [batch, n_rows] */
    uint16_t* out;              /* decode output: row r at out + (r - out_row0) * out_ld */
    int64_t out_ld, out_row0;   /*   (k_cols and 0, except for the chunks of the prefill GEMM) */
    int64_t n_rows, k_cols, k_pad;
    int64_t n_tiles, tile_begin;
    int64_t records_bytes;
    int32_t steps, atomic_y;
    int32_t last_steps;         /* symbols per lane of the last tile */
    uint32_t rec16;             /* records region size in 16-byte units */
    int64_t d_row;              /* GEMV: rows and columns a warp's next tile lies past */
    int64_t d_col;              /*   its current one (the launch's warps x tile width) */
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
    int sub_words;              /* hierarchical sub-table words staged in shared memory */
    /* x in tensor memory (batch 1, tiles inside rows, one tile width): TMEM lane l of
     * every warp's lane quarter holds, for each tile column c of a row, the x of the
     * columns lane l decodes in such a tile, 4 words per 8 symbols.  tx_cols = 0: x
     * is read from shared memory. */
    int tx_cols;                /* TMEM columns allocated (a power of 2 >= 32) */
    int tx_layout_cols;         /* columns per tile column: steps / 2 */
    int tx_used;                /* columns written: tile columns x tx_layout_cols */
    uint32_t tx_T;              /* tile width, 32 * steps */
};

struct HuffDecodeArgs {
    HuffMat m[kMaxDecodeBatch];
    int count;
    int64_t total_tiles;
    int* status;
    int code_bytes;
    int sub_words;              /* staged sub-table words (the largest single matrix's) */
};

/* Tensor-core GEMV launch (matrices whose tiles never cross a row).  A work item
 * is `rows` consecutive rows (one per decoding warp) x one tile column of a
 * matrix; items are numbered matrix by matrix, row block by row block, tile
 * column fastest. */
struct HuffMmaArgs {
    CUtensorMap xmap;                   /* x [batch, k_cols] BF16: boxes of 32 rows x 64 columns, 128-byte swizzle */
    HuffMat m[EC_MAX_GROUP];
    int count;
    int batch;                          /* rows of x in this pass, 1..kMmaMaxBatch */
    int* status;
    int code_bytes;                     /* per-warp code buffer */
    int64_t total_tiles;
    int64_t item_begin[EC_MAX_GROUP + 1];
    int32_t row_tiles[EC_MAX_GROUP];    /* tiles per row */
    uint32_t idesc;                     /* tcgen05 instruction descriptor (M = 64, N = warps) */
    int nbuf;                           /* chunk buffers (2 or 3) */
    int pool_bytes;                     /* one item's packed code areas, with slack */
    int sub_words;                      /* hierarchical sub-table words staged in shared memory */
};

/* ---- not in the Huffman GEMV: begin ---- */
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
    int32_t last_steps;         /* symbols per lane of the last tile */
    uint32_t rec16;             /* records region size in 16-byte units */
    int32_t tuple;              /* codes per symbol: 1 or 2 */
    int32_t values;             /* EC_RANS_VALUES_*: a 4-bit symbol s is the integer s - 8, or an FP4 E2M1 pattern */
};

struct RansArgs {
    RansMat m;
    int batch;
    const uint16_t* x;
    int* status;
};
/* ---- not in the Huffman GEMV: end ---- */

/* An FP8 matrix: rANS tiles of top-t table symbols plus per-tile correction records. */
struct Fp8Mat {
    const uint8_t* records;
    const uint32_t* tile_off;
    const uint32_t* table;      /* 2^prob_bits slot entries, 256 symbol values, 256 code values (FP32) */
    const float* row_scales;    /* [n_rows] */
    const uint32_t* esc_off;    /* [n_tiles + 1] record index */
    const uint32_t* esc;        /* position in the tile | code << 16 */
    float* y;
    uint16_t* out;
    int64_t n_rows, k_cols, k_pad;
    int64_t n_tiles;
    int64_t records_bytes;
    int32_t steps, prob_bits, atomic_y, words_cap;
    int32_t last_steps;
    uint32_t rec16;
};

struct Fp8Args {
    Fp8Mat m;
    int batch;
    const uint16_t* x;
    int* status;
};

/* A BF16 matrix whose exponents are rANS symbols under a top-t table (kind 5). */
struct ExpMat {
    const uint8_t* records;
    const uint32_t* tile_off;
    const uint32_t* table;      /* 2^prob_bits slot entries, then 256 exponent pairs */
    const uint8_t* raw;         /* sign / mantissa bytes, raw_tile bytes per tile */
    const uint32_t* esc_off;    /* [n_tiles + 1] record index */
    const uint32_t* esc;        /* position in the tile | BF16 pattern << 16 */
    float* y;
    uint16_t* out;
    int64_t n_rows, k_cols, k_pad;
    int64_t n_tiles;
    int64_t records_bytes;
    int32_t steps, prob_bits, atomic_y, words_cap;
    int32_t last_steps;
    uint32_t rec16;
    int32_t raw_tile;
    int32_t tuple;              /* exponents per symbol: 1 or 2 */
};

struct ExpArgs {
    ExpMat m;
    int batch;
    const uint16_t* x;
    int* status;
};

/* E8 lattice matrix (decode only). */
struct E8Mat {
    const uint8_t* records;
    const uint32_t* tile_off;
    const uint32_t* fc;         /* 17 x 32: freq | cum << 16 */
    const uint8_t* slot_sym;    /* 17 x 2^prob_bits: slot -> symbol */
    const float* row_scales;    /* [n_rows] */
    void* out;                  /* [n_rows, k_cols] BF16, FP8 E4M3 or INT8 */
    int64_t n_rows, k_cols, k_pad;
    int64_t n_tiles;
    int64_t records_bytes;
    int32_t steps, prob_bits, words_cap;
    int32_t last_steps;         /* vectors per lane of the last tile */
    uint32_t rec16;
    float scale;                /* the shared scale s */
};

struct E8Args {
    E8Mat m;
    int* status;
    int nbuf; /* tile buffers per warp: 2 (prefetch the next tile while decoding) or 1 */
};

/* ------------------------------------------------------------ small helpers */
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}

__device__ __forceinline__ void flag_corrupt(int* status) { atomicOr(status, 1); }

/* A read-only global load issued where it stands: loads that run a tile ahead of
 * their use must not be moved next to the use by the compiler, or their latency
 * comes back. */
__device__ __forceinline__ uint32_t ldg_early(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

/* Which matrix of a launch owns combined tile index g (count is small). */
template <class Args>
__device__ __forceinline__ int owner(const Args& a, int64_t g) {
    int k = 0;
    while (k + 1 < a.count && g >= a.m[k + 1].tile_begin) ++k;
    return k;
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
 * symbols i = 0 .. S-1 at positions 256 (i / 8) + 8 l + (i % 8), so every 8
 * symbols of a lane are 8 consecutive columns.  Each lookup of the pair table
 * (shared memory, indexed by the next EC_L1_BITS bits of the lane's stream)
 * yields exactly two exponents, already sitting in the BF16 exponent fields of a
 * 32-bit word [w(i+1) | w(i)].  With a fixed two symbols per lookup the decoded
 * exponents stay in registers at compile-time positions: one byte permute and one
 * bitwise select merge them with the raw sign/mantissa bytes
 *     bf16 = (sign << 15) | (exponent << 7) | mantissa     (DFloat11 Algorithm 1)
 * and the pair goes straight into the FP32 multiply-accumulate (GEMV) or to the
 * output (decode).  A window whose two codewords do not both fit takes a second
 * lookup for the second one (about 0.5% of lookups for LLM exponent statistics),
 * and a codeword longer than the window walks the hierarchical table in global
 * memory.
 *
 * Streams per warp: the lane starts and code area of the warp's next tile are
 * copied with cp.async into the second of two shared-memory buffers while the
 * current tile is decoded from the first; the raw bytes arrive with one
 * coalesced 16-byte load per lane per 16 symbols, two blocks ahead of use and
 * continuing into the next tile; x sits in shared memory as it is in memory
 * (rows of k_pad columns), and lane l reads the x of its 8 columns as one
 * 16-byte load (the 32 lanes read 512 contiguous bytes).
 */
constexpr int kMaxHW = 32;                     /* max warps per CTA */
/* After a code area: a lane whose data is corrupt may read up to 24 words past the
 * clamp point of its block (8 pairs, at most three word crossings each) */
constexpr int kSlackBytes = 128;
constexpr uint32_t kPairTabBytes = 4u * EC_PAIR_WORDS;
constexpr uint32_t kSignMant = 0x807F807Fu;    /* sign and mantissa bits of two BF16 */
constexpr int kSubSmemTables = 8;             /* hierarchical sub-tables staged in shared memory per launch */

__host__ __device__ constexpr int huff_max_warps(int b) { return b <= 1 ? 28 : (b <= 4 ? 24 : 16); }

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
    return v;
}
__device__ __forceinline__ uint32_t lds16(uint32_t a) {
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a) : "memory");
    return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a) : "memory");
    return v;
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

/* Tensor memory (TMEM) access of a warp: its 32 lanes are TMEM lanes 32 (warp % 4)
 * .. + 31 of the address's lane field; x4 = four consecutive 32-bit columns. */
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_ld4(uint32_t taddr, uint32_t (&v)[4]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
                 : "r"(taddr)
                 : "memory");
}
__device__ __forceinline__ void tc_ld8(uint32_t taddr, uint32_t (&v)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
                 : "r"(taddr)
                 : "memory");
}
__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tc_st4(uint32_t taddr, const uint4& v) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}
__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
/* Wait for this thread's TMEM loads; v (a load's destination) is tied to the wait
 * so that no use of it can be scheduled before the data is there. */
__device__ __forceinline__ void tc_wait_ld_into(uint32_t (&v)[4]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;" : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3])::"memory");
}
__device__ __forceinline__ void tc_wait_ld_into(uint32_t (&v)[8]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]), "+r"(v[6]), "+r"(v[7])::"memory");
}

/*
 * A lane's bit reader.  The lane's codewords sit LSB first in the staged code
 * area; A is the area bit where its next codeword starts.  The lane holds the two
 * area words lo, hi that cover bits S = A - 2 .. S + 63 (word index floor(S / 32)
 * and the next), so that
 *     v = funnel-shift-right(lo, hi, S mod 32)
 * has the stream's next 12 bits at bits 2..13 and v & 0x3FFC is already the byte
 * offset of their pair-table entry: one shift and one mask per lookup.
 * P accumulates whole table entries: only its low 5 bits (S mod 32, all the funnel
 * shift reads) and bit 5 matter.  An entry's bits 0..3 hold its advance and bits
 * 4..6 are 0, so bit 5 of P flips exactly when S crosses into the next word; then
 * lo takes hi, hi takes nx (the word after hi, loaded one crossing ahead so that
 * the next lookup never waits for a load) and nx the word at wa.  Hierarchical
 * launches, whose long codewords may cross several words, make that move at every
 * step (lane_adv); the others look past lo at most once per two steps and move
 * the window after every second step (pair_first, pair_second, lane_rebase).
 */
struct Lane {
    uint32_t P, lo, hi, nx, wa;
};

/* Position the lane at area bit A (a byte boundary); the two words before the area
 * (its lane starts) are readable, so A = 0 is fine. */
__device__ __forceinline__ void lane_seek(Lane& s, uint32_t area, uint32_t A) {
    const int32_t S = (int32_t)A - 2;
    const uint32_t a = area + (uint32_t)((S >> 5) * 4);
    s.lo = lds32(a);
    s.hi = lds32(a + 4);
    s.nx = lds32(a + 8);
    s.wa = a + 12;
    s.P = (uint32_t)S & 31u;
}

/* Pair-table entry of the window held in v (the next 12 stream bits at bits 2..13). */
__device__ __forceinline__ uint32_t pair_addr(uint32_t tab, uint32_t v) { return tab + (v & 0x3FFCu); }
/* Stage the 4096-entry pair table src into shared memory at dst. */
__device__ __forceinline__ void stage_pair_table(uint32_t* dst, const uint32_t* src) {
    for (int i = threadIdx.x; i < EC_PAIR_WORDS / 4; i += blockDim.x) ((uint4*)dst)[i] = __ldg((const uint4*)src + i);
}

/* Advance by the low bits of `e` (an entry, or a length below 32). */
__device__ __forceinline__ void lane_adv(Lane& s, uint32_t e) {
    const uint32_t pn = s.P + e;
    asm volatile(
        "{\n\t.reg .pred q;\n\t.reg .b32 t;\n\t"
        "lop3.b32 t, %4, %5, 32, 0x28;\n\t" /* (pn ^ P) & 32 */
        "setp.ne.u32 q, t, 0;\n\t"
        "@q mov.b32 %0, %1;\n\t"
        "@q mov.b32 %1, %2;\n\t"
        "@q ld.shared.u32 %2, [%3];\n\t"
        "@q add.u32 %3, %3, 4;\n\t}"
        : "+r"(s.lo), "+r"(s.hi), "+r"(s.nx), "+r"(s.wa)
        : "r"(pn), "r"(s.P)
        : "memory");
    s.P = pn;
}

/* Two steps without a data-dependent move on the lookup chain (non-hierarchical
 * launches).  At the start of a pair of steps (P & 32) = 0: the next codeword
 * starts at bit P mod 32 of lo.  Advances are at most 15 bits, so the second
 * step starts below bit 47 of lo, hi, nx and reads hi, nx when it is past lo;
 * after it, lane_rebase moves the window on by a word when the reader has left lo.
 * The chain from one lookup to the next is then shift, mask, add, load and the
 * advance (plus a select every second step) instead of also testing for and
 * making the move at every step. */
__device__ __forceinline__ uint32_t pair_first(Lane& s, uint32_t tab) {
    const uint32_t e = lds32(pair_addr(tab, __funnelshift_r(s.lo, s.hi, s.P)));
    s.P += e;
    return e;
}
__device__ __forceinline__ uint32_t pair_second(Lane& s, uint32_t tab) {
    const uint32_t v = (s.P & 32u) ? __funnelshift_r(s.hi, s.nx, s.P) : __funnelshift_r(s.lo, s.hi, s.P);
    const uint32_t e = lds32(pair_addr(tab, v));
    s.P += e;
    return e;
}
__device__ __forceinline__ void lane_rebase(Lane& s) {
    asm volatile(
        "{\n\t.reg .pred q;\n\t.reg .b32 t;\n\t"
        "and.b32 t, %4, 32;\n\t"
        "setp.ne.u32 q, t, 0;\n\t"
        "@q mov.b32 %0, %1;\n\t"
        "@q mov.b32 %1, %2;\n\t"
        "@q ld.shared.u32 %2, [%3];\n\t"
        "@q add.u32 %3, %3, 4;\n\t}"
        : "+r"(s.lo), "+r"(s.hi), "+r"(s.nx), "+r"(s.wa)
        : "r"(s.P)
        : "memory");
    s.P &= ~32u;
}

/* Area bit of the lane's next codeword. */
__device__ __forceinline__ uint32_t lane_pos(const Lane& s, uint32_t area) { return 8u * (s.wa - area) - 94u + (s.P & 31u); }

/* Keep the lane's loads inside the area and its slack (corrupt data only ever
 * moves wa past `limit`; the lane then decodes garbage, which the end-of-tile
 * check reports). */
__device__ __forceinline__ void lane_clamp(Lane& s, uint32_t limit) { s.wa = min(s.wa, limit); }

/* Hierarchical decoding context of the warp's current matrix (kHier launches). */
struct HierCtx {
    const uint32_t* sub; /* sub-tables (shared or global memory), 256 entries each */
    int n_sub;
    int* status;
};

/* A codeword longer than the window (or none, for corrupt data): walk the
 * sub-tables from the pair entry's sub-table index with the 30 stream bits w (the
 * codeword's first bit at bit 0).  Returns (exponent, length); corrupt data gives
 * exponent 0 of length 1 and sets the status. */
__device__ __forceinline__ uint2 long_codeword(uint32_t w, uint32_t ent, const HierCtx& h) {
    uint32_t t = (ent >> 7) & 0x1FFu, used = EC_L1_BITS, e = EC_ENT_BAD;
#pragma unroll 1
    for (int lvl = 0; lvl < 2; ++lvl) {
        if ((int)t >= h.n_sub || used > 22) {
            e = EC_ENT_BAD;
            break;
        }
        e = h.sub[256 * t + ((w >> used) & 0xFFu)];
        if (!(e & EC_ENT_PTR) || (e & EC_ENT_BAD)) break;
        t = e & 0xFFFFu;
        used = (e >> 16) & 31u;
    }
    if (e & (EC_ENT_PTR | EC_ENT_BAD) || ((e >> 16) & 31u) > 30u || ((e >> 16) & 31u) == 0u) {
        flag_corrupt(h.status);
        return make_uint2(0u, 1u);
    }
    return make_uint2((e & 0xFFFFu) >> 7, (e >> 16) & 31u);
}

/* An open pair entry e (hierarchical launches): the lane has already advanced by
 * the first codeword when it fits the window; decode what is missing and return
 * the pair's exponents in BF16 position [e1 << 23 | e0 << 7]. */
__device__ __forceinline__ uint32_t pair_open(Lane& s, uint32_t e, uint32_t tab, const HierCtx& h) {
    uint32_t e0 = (e >> 7) & 0xFFu;
    if (((e >> EC_PAIR_FIRST_SHIFT) & 15u) == 0) {
        const uint2 r = long_codeword(__funnelshift_r(s.lo, s.hi, s.P) >> 2, e, h);
        e0 = r.x;
        lane_adv(s, r.y);
    }
    const uint32_t f = lds32(pair_addr(tab, __funnelshift_r(s.lo, s.hi, s.P)));
    uint32_t e1 = (f >> 7) & 0xFFu, l1 = (f >> EC_PAIR_FIRST_SHIFT) & 15u;
    if (l1 == 0) {
        const uint2 r = long_codeword(__funnelshift_r(s.lo, s.hi, s.P) >> 2, f, h);
        e1 = r.x;
        l1 = r.y;
    }
    lane_adv(s, l1);
    return (e0 << 7) | (e1 << 23);
}

/* The lane's next two symbols: their exponents in BF16 position [e(i+1) << 23 |
 * e(i) << 7] (other bits unspecified).  Without kHier the encoder guarantees every
 * pair fits the window (window records), so a step is one shift, one mask, one
 * table load and the advance, with no branch on the data. */
template <bool kHier>
__device__ __forceinline__ uint32_t pair_step(Lane& s, uint32_t tab, const HierCtx& h) {
    const uint32_t e = lds32(pair_addr(tab, __funnelshift_r(s.lo, s.hi, s.P)));
    lane_adv(s, e);
    if (kHier && __builtin_expect((int32_t)e < 0, 0)) return pair_open(s, e, tab, h);
    return e;
}

/* (r & 0x807F807F) | (e & ~0x807F807F) in one instruction. */
__device__ __forceinline__ uint32_t merge_sm(uint32_t r, uint32_t e) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xE4;" : "=r"(d) : "r"(r), "r"(e), "n"(kSignMant));
    return d;
}

/* Eight symbols of the lane (raw words r0 = symbols 0..3, r1 = 4..7) as four
 * words [w(i+1) | w(i)]. */
template <bool kHier>
__device__ __forceinline__ void decode8(Lane& s, uint32_t tab, const HierCtx& h, uint32_t r0, uint32_t r1,
                                        uint32_t (&w)[4]) {
    if (!kHier) {
        const uint32_t e0 = pair_first(s, tab);
        const uint32_t e1 = pair_second(s, tab);
        lane_rebase(s);
        w[0] = merge_sm(r0, e0);
        w[1] = merge_sm(__funnelshift_r(r0, r0, 8), e1);
        const uint32_t e2 = pair_first(s, tab);
        const uint32_t e3 = pair_second(s, tab);
        lane_rebase(s);
        w[2] = merge_sm(r1, e2);
        w[3] = merge_sm(__funnelshift_r(r1, r1, 8), e3);
        return;
    }
    const uint32_t e0 = pair_step<kHier>(s, tab, h);
    const uint32_t e1 = pair_step<kHier>(s, tab, h);
    w[0] = merge_sm(r0, e0);
    w[1] = merge_sm(__funnelshift_r(r0, r0, 8), e1);
    const uint32_t e2 = pair_step<kHier>(s, tab, h);
    const uint32_t e3 = pair_step<kHier>(s, tab, h);
    w[2] = merge_sm(r1, e2);
    w[3] = merge_sm(__funnelshift_r(r1, r1, 8), e3);
}

/* A window record (13-bit tile position | sign and mantissa << 13 | exponent << 21):
 * the BF16 weight with exponent `expo` (the record's own, or the coded one). */
__device__ __forceinline__ uint32_t rec_weight(uint32_t r, uint32_t expo) {
    return ((r >> (EC_HREC_SM_SHIFT + 7 - 15)) & 0x8000u) | (expo << 7) | ((r >> EC_HREC_SM_SHIFT) & 0x7Fu);
}
__device__ __forceinline__ uint32_t rec_pos(uint32_t r) { return r & EC_HREC_POS_MASK; }
__device__ __forceinline__ uint32_t rec_exp(uint32_t r) { return r >> EC_HREC_EXP_SHIFT; }

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
/* acc0 += w0 * x0, acc1 += w1 * x1 (two chains). */
__device__ __forceinline__ void fma2x_bf16(uint32_t w, uint32_t x, float& acc0, float& acc1) {
    asm("{\n\t.reg .b16 wl, wh, xl, xh;\n\t"
        "mov.b32 {wl, wh}, %2;\n\t"
        "mov.b32 {xl, xh}, %3;\n\t"
        "fma.rn.f32.bf16 %0, wl, xl, %0;\n\t"
        "fma.rn.f32.bf16 %1, wh, xh, %1;\n\t}"
        : "+f"(acc0), "+f"(acc1)
        : "r"(w), "r"(x));
}
/* acc += w * x for one BF16 weight and one BF16 activation (low halves). */
__device__ __forceinline__ float fma1_bf16(uint32_t w, uint32_t x, float acc) {
    asm("{\n\t.reg .b16 wl, wh, xl, xh;\n\t"
        "mov.b32 {wl, wh}, %1;\n\t"
        "mov.b32 {xl, xh}, %2;\n\t"
        "fma.rn.f32.bf16 %0, wl, xl, %0;\n\t}"
        : "+f"(acc)
        : "r"(w), "r"(x));
    return acc;
}

__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;"); }

/* Per-warp shared memory: two tile buffers, each the 64 bytes of lane starts, the
 * code area and slack, then the two buffers' mbarriers (8 bytes each).  Multiples
 * of 16 bytes when code_bytes is. */
__host__ __device__ constexpr size_t tile_buf_bytes(int code_bytes) { return 64 + (size_t)code_bytes + kSlackBytes; }
__host__ __device__ constexpr size_t huff_warp_bytes(int code_bytes) { return 2 * tile_buf_bytes(code_bytes) + 16; }
static_assert(kSlackBytes % 16 == 0 && kSlackBytes >= 8 * 48 / 8 + 16 && kPairTabBytes % 16 == 0, "alignment");
static_assert(huff_warp_bytes(16) % 16 == 0 && huff_warp_bytes(4112) % 16 == 0, "per-warp block alignment");

/* x for the GEMV: per batch row, k_pad BF16 values (zero past K). */
__host__ __device__ constexpr size_t xs_row_bytes(uint32_t kp) { return (size_t)2 * kp; }

/* Stage x [batch, K] (BF16) into shared rows of k_pad entries, zero past K:
 * 16-byte loads and stores, four in flight per thread, when K % 8 == 0. */
__device__ __forceinline__ void stage_x_rows(uint16_t* xs, const uint16_t* __restrict__ x, int batch, int64_t K,
                                             uint32_t kp) {
    if ((K & 7) == 0) {
        const uint32_t per_row = kp / 8, n = (uint32_t)batch * per_row;
        for (uint32_t i0 = threadIdx.x; i0 < n; i0 += 4 * blockDim.x) {
            uint4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const uint32_t i = i0 + u * blockDim.x, b = i / per_row, c = (i - b * per_row) * 8;
                v[u] = i < n && c < K ? __ldg((const uint4*)(x + (int64_t)b * K + c)) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const uint32_t i = i0 + u * blockDim.x;
                if (i < n) *(uint4*)(xs + (size_t)i * 8) = v[u];
            }
        }
    } else {
        for (int b = 0; b < batch; ++b)
            for (uint32_t c = threadIdx.x; c < kp; c += blockDim.x) xs[(size_t)b * kp + c] = c < K ? x[b * K + c] : 0;
    }
}

/* A resolved tile record (all lanes hold the same values). */
struct TileRef {
    const uint8_t* rec; /* lane starts | raw | code area */
    uint32_t t;         /* tile index within its matrix (a launch has < 2^31 tiles) */
    int mi;             /* matrix of the launch */
    int S;              /* symbols per lane */
    int area;           /* bytes of window records + code area; 0 = corrupt record (skipped) */
};

template <class Args>
__device__ __forceinline__ uint2 tile_offsets_of(const Args& a, int64_t g, int mi) {
    const HuffMat& M = a.m[mi];
    const int64_t t = g - M.tile_begin;
    return make_uint2(ldg_early(M.tile_off + t), ldg_early(M.tile_off + t + 1));
}
template <class Args>
__device__ __forceinline__ uint2 tile_offsets(const Args& a, int64_t g) {
    return tile_offsets_of(a, g, owner(a, g));
}

/* Resolve combined tile g from its record offsets (16-byte units); a record whose
 * extent is inconsistent gets area 0. */
template <class Args>
__device__ __forceinline__ TileRef tile_ref_of(const Args& a, int64_t g, uint2 off, int mi) {
    TileRef r;
    r.mi = mi;
    const HuffMat& M = a.m[r.mi];
    r.t = (uint32_t)(g - M.tile_begin);
    r.S = r.t == M.n_tiles - 1 ? M.last_steps : M.steps;
    /* offsets are 16-byte units; a record is far below 4 GB */
    const int area = (int)((off.y - off.x) * 16u) - 64 - EC_RAW_BYTES(r.S);
    const bool ok = off.x <= off.y && off.y <= M.rec16 && area >= 16;
    r.rec = M.records + (size_t)(ok ? off.x : 0u) * 16;
    r.area = ok ? area : 0;
    return r;
}
template <class Args>
__device__ __forceinline__ TileRef tile_ref(const Args& a, int64_t g, uint2 off) {
    return tile_ref_of(a, g, off, owner(a, g));
}

/* mbarrier and bulk-copy helpers (one arrival per phase: the issuing lane's). */
__device__ __forceinline__ void mbar_init(uint32_t mbar) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(mbar) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(uint32_t mbar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(mbar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t mbar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(mbar)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t mbar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(mbar), "r"(parity)
        : "memory");
    return ok != 0;
}
/* Wait for phase `parity` of mbar with a bound on the attempts (each of which may
 * suspend the thread for a while); false when the bound ran out. */
__device__ __forceinline__ bool mbar_wait(uint32_t mbar, uint32_t parity) {
    for (int i = 0; i < (1 << 20); ++i)
        if (mbar_try_wait(mbar, parity)) return true;
    return false;
}

/* Start the copy of a tile's lane starts (64 bytes) and code area into a tile
 * buffer: one lane arms the buffer's mbarrier with the byte count and issues two
 * bulk copies (16-byte aligned, multiples of 16 bytes); a corrupt record only
 * arrives, so the phase still completes. */
__device__ __forceinline__ void prefetch_code(uint32_t buf, uint32_t mbar, const TileRef& r, int lane, int cap) {
    if (lane == 0) {
        if (r.area > 0) {
            const uint32_t n = (uint32_t)min(r.area, cap); /* the code area, then as many records as fit */
            mbar_arrive_tx(mbar, 64u + n);
            bulk_g2s(buf, r.rec, 64u, mbar);
            bulk_g2s(buf + 64, r.rec + 64 + EC_RAW_BYTES(r.S), n, mbar);
        } else {
            mbar_arrive_tx(mbar, 0u);
        }
    }
}

/* Decoding context of one matrix of a launch: its pair table in shared memory and,
 * for hierarchical launches, its sub-tables. */
struct WalkCtx {
    uint32_t tab;
    HierCtx h;
};

/* Sub-tables of matrix M: staged in shared memory (`staged`, the launch's block of
 * them) when the launch staged them, else read from the blob. */
__device__ __forceinline__ HierCtx hier_ctx(const HuffMat& M, const uint32_t* staged, int* status) {
    HierCtx h;
    h.sub = M.sub_smem >= 0 ? staged + M.sub_smem : M.table + EC_PAIR_WORDS;
    h.n_sub = M.n_sub;
    h.status = status;
    return h;
}

/* Stage the launch's sub-tables that fit (kSubSmemTables in all) into shared memory. */
template <class Args>
__device__ __forceinline__ void stage_sub_tables(const Args& a, uint32_t* dst) {
    for (int k = 0; k < a.count; ++k) {
        const HuffMat& M = a.m[k];
        if (M.sub_smem < 0) continue;
        const uint4* src = (const uint4*)(M.table + EC_PAIR_WORDS);
        uint4* d = (uint4*)(dst + M.sub_smem);
        for (int i = threadIdx.x; i < 64 * M.n_sub; i += blockDim.x) d[i] = __ldg(src + i);
    }
}

/* Layout of a staged tile: its buffer holds the 64 bytes of lane starts (lane 0's
 * slot: the window record count n), the code area, and the records as far as the
 * buffer's room `cap` allows; the rest stay in the tile record in global memory. */
struct TileRecs {
    int n;          /* window records; -1: inconsistent counts (corrupt data) */
    uint32_t code;  /* code area bytes */
    uint32_t staged; /* records in the buffer, after the code area */
};
__device__ __forceinline__ TileRecs tile_recs(uint32_t buf, int area, int cap) {
    TileRecs t;
    t.n = (int)lds16(buf);
    const int code = area - 16 * ((4 * t.n + 15) / 16);
    if (area <= 0 || code < 16 || code > cap) {
        t.n = -1;
        t.code = t.staged = 0;
        return t;
    }
    t.code = (uint32_t)code;
    t.staged = (uint32_t)min(t.n, (min(area, cap) - code) / 4);
    return t;
}
/* Where the tile's records beyond the staged ones sit in global memory. */
__device__ __forceinline__ const uint32_t* far_records(const TileRef& r, uint32_t code) {
    return (const uint32_t*)(r.rec + 64 + EC_RAW_BYTES(r.S) + code);
}

/* Walk combined tiles g0, g0 + stride, ... < g_end.  The first tile's copy must
 * already be in flight (prefetch_code).  For every tile with a sound record:
 * begin(tile) once; then, for each block of 16 symbols of the lane, block(buf,
 * tile) and two calls half(w, h) for its two 8-symbol halves h = 0, 1 in order (w =
 * four words [w(i+1) | w(i)]); then end(tile, buf, recs).  buf is the tile's shared
 * buffer: lane starts, the code area, then its window records (tile_recs).  Rows start on block boundaries (k_pad is
 * a multiple of 16 * 32 positions).  The raw bytes of block b + 2 are loaded right
 * after block b is decoded, into the ring slot it frees; blocks 0 and 1 of the
 * next tile are loaded the same way at the end of the current one. */
template <bool kHier, class Args, class CtxOf, class Begin, class Block, class Half, class End>
__device__ __forceinline__ void huff_walk(const Args& a, uint32_t g0, uint32_t stride, uint32_t g_end, TileRef cur,
                                          uint32_t bufs, uint32_t buf_bytes, uint32_t& ph, int lane,
                                          CtxOf&& ctx_of, Begin&& begin, Block&& block, Half&& half, End&& end) {
    const uint32_t mbars = bufs + 2 * buf_bytes;
    int mi_next = g0 + stride < g_end ? owner(a, g0 + stride) : 0; /* matrix of the next tile */
    uint2 off_next = g0 + stride < g_end ? tile_offsets_of(a, g0 + stride, mi_next) : make_uint2(0u, 0u);
    uint4 rr[2] = {};
    bool raw_ready = false, raw_swap = false;
    uint32_t cb = bufs; /* buffer of the current tile */
    for (uint32_t g = g0; g < g_end; g += stride) {
        const uint32_t bi = cb == bufs ? 0u : 1u;
        const bool arrived = mbar_wait(mbars + 8 * bi, (ph >> bi) & 1u); /* the current tile's copy */
        ph ^= 1u << bi;
        __syncwarp(); /* every lane is done with the other buffer */
        if (!arrived) cur.area = 0; /* (never seen: the copy did not complete in time) */
        const uint32_t nb_buf = cb == bufs ? bufs + buf_bytes : bufs; /* the next tile's buffer */
        const bool has_next = g + stride < g_end;
        TileRef nxt{};
        if (has_next) {
            nxt = tile_ref_of(a, g + stride, off_next, mi_next);
            prefetch_code(nb_buf, mbars + 8 * (bi ^ 1u), nxt, lane, a.code_bytes);
            if (g + 2 * stride < g_end) {
                mi_next = owner(a, g + 2 * stride);
                off_next = tile_offsets_of(a, g + 2 * stride, mi_next);
            }
        }
        const TileRecs tr = tile_recs(cb, cur.area, a.code_bytes);
        if (tr.n < 0) {
            if (lane == 0) flag_corrupt(a.status);
            raw_ready = false;
            cur = nxt;
            cb = nb_buf;
            continue;
        }
        const uint32_t cbytes = tr.code;
        const uint32_t s0 = lane ? lds16(cb + 2 * lane) : 0u;
        const uint32_t s1 = lane < 31 ? lds16(cb + 2 * lane + 2) : 0u;
        const WalkCtx c = ctx_of(cur.mi);
        const uint32_t area = cb + 64;
        const uint4* raw4 = (const uint4*)(cur.rec + 64) + lane;
        const int nb = cur.S / 16;
        const uint32_t limit = area + cbytes;
        Lane s;
        lane_seek(s, area, 8u * min(s0, cbytes));
        if (!raw_ready) {
            rr[0] = __ldg(raw4);
            if (nb > 1) rr[1] = __ldg(raw4 + 32);
        } else if (raw_swap) { /* the previous tile's block count was odd */
            const uint4 t = rr[0];
            rr[0] = rr[1];
            rr[1] = t;
        }
        /* each decoded block's slot takes the block two ahead, continuing into blocks
         * 0 and 1 of the next tile; after an odd block count those land in slots 1
         * and 0 and are swapped when the next tile starts */
        const bool chain = has_next && nxt.area > 0 && nb >= 2;
        const uint4* nraw4 = (const uint4*)((chain ? nxt.rec : cur.rec) + 64) + lane;
        const int nnbc = chain ? min(2, nxt.S / 16) : 0; /* next-tile blocks to prefetch */
        begin(cur);
        for (int b0 = 0; b0 < nb; b0 += 2) {
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int blk = b0 + u;
                if (u == 0 || blk < nb) {
                    block(cb, cur);
                    lane_clamp(s, limit);
                    uint32_t w[4];
                    decode8<kHier>(s, c.tab, c.h, rr[u].x, rr[u].y, w);
                    half(w, 0);
                    decode8<kHier>(s, c.tab, c.h, rr[u].z, rr[u].w, w);
                    half(w, 1);
                    const int ahead = blk + 2;
                    if (ahead < nb) rr[u] = __ldg(raw4 + 32 * ahead);
                    else if (ahead - nb < nnbc) rr[u] = __ldg(nraw4 + 32 * (ahead - nb));
                }
            }
        }
        raw_ready = chain;
        raw_swap = chain && (nb & 1);
        /* every lane's codewords end in the last byte before the next lane's start
         * (the last lane: before the >= 8 zero bytes closing the area) */
        const uint32_t p = lane_pos(s, area), pmax = 8u * cbytes;
        const bool bad = lane < 31 ? (p > 8u * s1 || p + 8u <= 8u * s1) : (p + 64u > pmax);
        if (__any_sync(kFull, bad) && lane == 0) flag_corrupt(a.status);
        end(cur, cb, tr);
        cur = nxt;
        cb = nb_buf;
    }
}

/* Records j in [from, n) of a tile, read from global memory (those the tile buffer
 * had no room for): the lane's share of sum (w - w_coded) * x over the records at
 * tile positions [lo, hi), x[column] at xrow + 2 (col_base + position).  Rare; its
 * loads are volatile so that they stay inside the branch that needs them. */
__device__ __forceinline__ float far_records_dot(const uint32_t* far, uint32_t from, uint32_t n, uint32_t lo, uint32_t hi,
                                              uint32_t col_base, uint32_t xrow, uint32_t fill, int lane) {
    float d = 0.f;
    for (uint32_t j = from + (uint32_t)lane; j < n; j += 32) {
        const uint32_t e = ldg_early(far + j), q = rec_pos(e);
        if (q >= lo && q < hi) {
            const uint32_t xv1 = lds16(xrow + 2u * (col_base + q));
            d = fma1_bf16(rec_weight(e, rec_exp(e)), xv1, d);
            d = fma1_bf16(rec_weight(e, fill) ^ 0x8000u, xv1, d);
        }
    }
    return d;
}

/* ======================================================== Huffman GEMV kernel */
/* kPart = false: row sums go to y (stored, or added atomically when a row spans
 * tiles).  kPart = true (allocation-free entry point): every row segment a tile
 * produces goes to its own slot of a.part, summed into y by part_reduce_kernel.
 * kHier: some matrix of the launch decodes through the hierarchical tables. */
template <int B, bool kPart, bool kHier, bool kTx>
__global__ void __launch_bounds__(huff_max_warps(B) * 32, 1) huff_gemv_kernel(const __grid_constant__ HuffGemvArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t kp = (uint32_t)a.m[0].k_pad;
    const int64_t K = a.m[0].k_cols;
    const int batch = a.batch;
    static_assert(!kTx || B == 1, "x in tensor memory: batch 1 only");

    /* shared: TMEM address (16 B) | pair tables | staged sub-tables | x [batch][k_pad] |
     * per warp: two tile buffers */
    const uint32_t tslot = smem_u32(smem);
    uint4* tabs = (uint4*)(smem + 16);
    uint32_t* subs = (uint32_t*)(smem + 16 + (size_t)a.count * kPairTabBytes);
    uint16_t* xs = (uint16_t*)(subs + a.sub_words);
    uint8_t* wbase = (uint8_t*)xs + (size_t)batch * xs_row_bytes(kp) + (size_t)warp * huff_warp_bytes(a.code_bytes);
    const uint32_t bufs = smem_u32(wbase), buf_bytes = (uint32_t)tile_buf_bytes(a.code_bytes);
    const uint32_t xs_s = smem_u32(xs), xs_lane = xs_s + 16u * lane, tabs_s = smem_u32(tabs); /* x of the lane's 8 columns */

    /* Warps are numbered CTA-fastest (warp w of CTA c is gw = w * grid + c) and take tiles
     * gw, gw + nw, ...: the tiles of one CTA lie spread over the whole launch, so every
     * CTA gets about the same number of code bytes even when a partial last round or
     * regions of longer codewords would load some CTAs more than others. */
    const int nwarp = blockDim.x >> 5;
    const int64_t gw = (int64_t)warp * gridDim.x + blockIdx.x, nw = (int64_t)gridDim.x * nwarp;
    const uint32_t mbars = bufs + 2 * buf_bytes;
    if (lane == 0) {
        mbar_init(mbars);
        mbar_init(mbars + 8);
        mbar_fence_init();
    }
    __syncwarp();
    uint32_t ph = 0; /* parity of the next phase of each buffer's mbarrier */
    TileRef first{};
    if (gw < a.total_tiles) {
        first = tile_ref(a, gw, tile_offsets(a, gw));
        prefetch_code(bufs, mbars, first, lane, a.code_bytes);
    }
    for (int k = 0; k < a.count; ++k) stage_pair_table((uint32_t*)(tabs + k * (EC_PAIR_WORDS / 4)), a.m[k].table);
    if (kHier) stage_sub_tables(a, subs);
    if (kTx && warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(tslot), "r"(a.tx_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    grid_dep_launch();
    grid_dep_wait(); /* x and y belong to the preceding kernel in the stream from here on */
    stage_x_rows(xs, a.x, batch, K, kp);
    uint32_t tx = 0; /* TMEM address of the warp's lane quarter, column 0 */
    if (kTx) {
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        tx = lds32(tslot) + ((uint32_t)(32 * (warp & 3)) << 16);
        if (warp < 4) { /* one warp per lane quarter writes the x layouts */
            for (uint32_t c = 0; c < (uint32_t)a.tx_used; c += 4) {
                const uint32_t L = c / (uint32_t)a.tx_layout_cols, m = (c - L * (uint32_t)a.tx_layout_cols) / 4;
                tc_st4(tx + c, lds128(xs_s + 2u * (L * a.tx_T + 256u * m + 8u * lane)));
            }
            tc_wait_st();
        }
        tc_fence_before();
    }
    __syncthreads();
    if (kTx) tc_fence_after();

    if (gw < a.total_tiles) {
    const uint32_t jrow = kp / 32;
    int prev_mi = -1;
    uint32_t prev_t = 0, row0 = 0, col0 = 0; /* where this warp's current tile starts (rows, columns < 2^31) */
    /* batch 1: four independent sums (two FMAs each per 8 symbols: products of the high
     * BF16 halves have the longer latency); wider batches two per row */
    constexpr int kAcc = B == 1 ? 4 : 2;
    float acc[B][kAcc];
    /* x of the current 8 symbols: loaded one half-block ahead for narrow batches,
     * at use for wide ones (whose registers go to the accumulators) */
    constexpr bool kAhead = B <= 4;
    uint4 xv[kAhead ? B : 1];
    /* kTx: x of the current 16 symbols (one decode block), loading from TMEM; the load
     * of the next block's is issued when a block's second half is done, whether or not
     * the tile has one (the allocation has 8 columns to spare) */
    uint32_t xt[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
    uint32_t xcol = 0; /* kTx: its TMEM address */
    uint32_t row = 0, t_cur = 0;
    uint32_t jc = 0; /* first column / 32 of the current 8 symbols' 256-column block */
    const HuffMat* Mp = &a.m[0];
    auto load_x = [&](uint32_t j) {
        const uint32_t xa = xs_lane + 64 * j;
#pragma unroll
        for (int b = 0; b < (kAhead ? B : 0); ++b) {
            if (B > 1 && b >= batch) break;
            xv[b] = lds128(xa + (uint32_t)(b * xs_row_bytes(kp)));
        }
    };
    /* Row r of the current tile (buffer cb) is complete: fold in its window records
     * (each adds (w - w_coded) * x, both products exact; they came with the tile's
     * code area, all but those beyond the buffer's room), then reduce across the warp. */
    auto flush = [&](uint32_t r, uint32_t cb, const TileRef& tile, const TileRecs& tr) {
        const HuffMat& M = *Mp;
        /* (with x in tensor memory every tile lies inside its row: r = row0, and every
         * record of the tile belongs to it) */
        const uint32_t seg_end = kTx ? ~0u : (r - row0 + 1) * kp - col0;    /* tile positions of rows <= r */
        const uint32_t seg_begin = kTx || r == row0 ? 0u : seg_end - kp;    /* ... of rows < r */
        const uint32_t col_base = kTx ? col0 : col0 - (r - row0) * kp;      /* column = col_base + position */
        for (uint32_t j = (uint32_t)lane; j < tr.staged; j += 32) {
            const uint32_t e = lds32(cb + 64 + tr.code + 4 * j), q = rec_pos(e);
            if (q >= seg_begin && q < seg_end) {
                const uint32_t col = col_base + q;
                const uint32_t wt = rec_weight(e, rec_exp(e));
                const uint32_t wf = rec_weight(e, (uint32_t)M.fill) ^ 0x8000u; /* minus the coded weight */
#pragma unroll
                for (int b = 0; b < B; ++b) {
                    if (B > 1 && b >= batch) break;
                    const uint32_t xv1 = lds16(xs_s + 2u * ((uint32_t)b * kp + col));
                    acc[b][0] = fma1_bf16(wt, xv1, acc[b][0]);
                    acc[b][0] = fma1_bf16(wf, xv1, acc[b][0]);
                }
            }
        }
        if (tr.n > (int)tr.staged) { /* (rare) records beyond the buffer's room */
            const uint32_t* far = far_records(tile, tr.code);
#pragma unroll
            for (int b = 0; b < B; ++b) {
                if (B > 1 && b >= batch) break;
                acc[b][0] += far_records_dot(far, tr.staged, (uint32_t)tr.n, seg_begin, seg_end, col_base,
                                             xs_s + 2u * (uint32_t)b * kp, (uint32_t)M.fill, lane);
            }
        }
        int64_t slot = 0;
        if (kPart) /* tiles before this one that also cover row r */
            slot = (int64_t)t_cur - ((int64_t)r * M.k_pad) / (32 * (int64_t)M.steps);
#pragma unroll
        for (int b = 0; b < B; ++b) {
            if (B > 1 && b >= batch) break;
            float t = acc[b][0];
#pragma unroll
            for (int j = 1; j < kAcc; ++j) t += acc[b][j];
            const float sum = warp_sum(t);
            if (lane == 0) {
                if (kPart) {
                    a.part[((int64_t)b * M.n_rows + r) * a.part_slots + slot] = sum;
                } else {
                    float* dst = M.y + (int64_t)b * M.n_rows + r;
                    if (M.atomic_y) atomicAdd(dst, sum);
                    else *dst = sum;
                }
            }
#pragma unroll
            for (int j = 0; j < kAcc; ++j) acc[b][j] = 0.f;
        }
    };
    huff_walk<kHier>(
        a, gw, nw, a.total_tiles, first, bufs, buf_bytes, ph, lane,
        [&](int mi) {
            WalkCtx c;
            c.tab = tabs_s + mi * kPairTabBytes;
            c.h = hier_ctx(a.m[mi], subs, a.status);
            return c;
        },
        [&](const TileRef& r) {
            Mp = &a.m[r.mi];
            t_cur = r.t;
            if (r.mi == prev_mi && r.t == prev_t + (uint32_t)nw) { /* the same matrix, the next tile of this warp */
                row0 += (uint32_t)Mp->d_row;
                col0 += (uint32_t)Mp->d_col;
                if (col0 >= kp) {
                    col0 -= kp;
                    ++row0;
                }
            } else {
                const int64_t T = 32 * (int64_t)Mp->steps;
                row0 = (uint32_t)tile_row(r.t, T, kp, EC_HUFF_ROW_ALIGN);
                col0 = (uint32_t)((int64_t)r.t * T - (int64_t)row0 * kp);
            }
            prev_mi = r.mi;
            prev_t = r.t;
            row = row0; /* advanced by the block hook as rows end inside the tile */
            if (!kTx) jc = (uint32_t)col0 / 32;
            if (kTx) {
                xcol = tx + col0 / 64u; /* (col0 / T) layouts of T / 64 columns; col0 is a multiple of T */
                tc_wait_ld_into(xt); /* the previous tile's last (unused) load */
                tc_ld8(xcol, xt);
            } else if (kAhead) {
                load_x(jc);
            }
#pragma unroll
            for (int b = 0; b < B; ++b)
#pragma unroll
                for (int j = 0; j < kAcc; ++j) acc[b][j] = 0.f;
        },
        [&](uint32_t cb, const TileRef& tile) {
            if (!kTx && jc >= jrow) { /* (with x in TMEM tiles lie inside rows) */
                flush(row, cb, tile, tile_recs(cb, tile.area, a.code_bytes));
                jc -= jrow;
                ++row;
            }
        },
        [&](const uint32_t (&w)[4], int h) {
            if (kTx && h == 0) tc_wait_ld_into(xt);
#pragma unroll
            for (int b = 0; b < B; ++b) {
                if (B > 1 && b >= batch) break;
                const uint4 x4 = kTx ? make_uint4(xt[4 * h % 8], xt[(4 * h + 1) % 8], xt[(4 * h + 2) % 8], xt[(4 * h + 3) % 8])
                                     : kAhead ? xv[b] : lds128(xs_lane + 64 * jc + (uint32_t)(b * xs_row_bytes(kp)));
                if (B == 1) {
                    fma2x_bf16(w[0], x4.x, acc[b][0], acc[b][1 % kAcc]);
                    fma2x_bf16(w[1], x4.y, acc[b][2 % kAcc], acc[b][3 % kAcc]);
                    fma2x_bf16(w[2], x4.z, acc[b][0], acc[b][1 % kAcc]);
                    fma2x_bf16(w[3], x4.w, acc[b][2 % kAcc], acc[b][3 % kAcc]);
                } else {
                    fma2x_bf16(w[0], x4.x, acc[b][0], acc[b][1]);
                    fma2x_bf16(w[1], x4.y, acc[b][0], acc[b][1]);
                    fma2x_bf16(w[2], x4.z, acc[b][0], acc[b][1]);
                    fma2x_bf16(w[3], x4.w, acc[b][0], acc[b][1]);
                }
            }
            if (!kTx) jc += 8;
            if (kTx) { /* the next 8 symbols' x, if the tile has them (one load in flight at a time) */
                if (h == 1) {
                    xcol += 8;
                    tc_ld8(xcol, xt);
                }
            } else if (kAhead) {
                /* rows start on block boundaries: only a second half can be followed by
                 * a new row */
                load_x(h == 1 && jc >= jrow ? jc - jrow : jc);
            }
        },
        [&](const TileRef& tile, uint32_t cb, const TileRecs& tr) { flush(row, cb, tile, tr); });
    }
    if (kTx) { /* every warp is done with tensor memory */
        tc_wait_ld(); /* the load past the warp's last block */
        tc_fence_before();
        __syncthreads();
        if (warp == 0) {
            tc_fence_after();
            asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(lds32(tslot)), "r"(a.tx_cols)
                         : "memory");
        }
    }
}

/* ---- not in the Huffman GEMV: begin ---- */
/* ========================================= Huffman tensor-core GEMV (tcgen05) */
/*
 * Small batches (MINE section 5: fused kernels for batch > 1 as the next step)
 * put the product on the 5th-generation tensor cores: y^T = X W^T with BF16
 * operands in shared memory and FP32 accumulators in tensor memory.
 *
 * Roles: warp 0 produces (x by TMA, the MMAs, a quarter of the read-out); warps
 * 1 .. rows decode, one weight row each (rows = warps - 1; N = warps, a multiple
 * of 8, the operand's last row unused).
 *
 * Work item: `rows` consecutive rows x one tile column, for matrices whose tiles
 * do not cross rows.  The item runs in chunks of 256 columns, 8 symbols of every
 * lane.  Lane l of a decoding warp decodes its 8 symbols (columns 8 l .. 8 l + 7
 * of the chunk) and stores them as ONE 16-byte row segment of a
 * 128-byte-swizzled K-major operand: chunk l % 8 of the 128-byte row in swizzle
 * atom l / 8, so the 32 stores of a warp hit all banks (4 wavefronts).  x arrives
 * by TMA in the same swizzled layout (boxes of 32 rows x 64 columns; rows past
 * the batch and columns past K read as zero), nbuf - 1 chunks ahead.  An item's
 * code areas (64 bytes of lane starts + the code area per row) are staged packed
 * in one of two pools, the next item's while this one is decoded.
 *
 * MMA: M = 64 rows of x (the batch; rows past it are never read back), N = warps
 * weight rows, K = 16, kind::f16 with BF16 inputs; 16 per chunk, issued by one
 * elected lane of the converged producer warp once every decoding warp has
 * stored the chunk (mbarrier `full`) and its x has landed (`xfull`), then
 * committed to the chunk buffer's mbarrier (`done`), which the decoders and the
 * next x copy wait on before reusing the buffer.  MMAs that accumulate into one
 * TMEM tile run one after the other, so a chunk spreads its 16 over four tiles
 * (k step mod 4) and consecutive chunks use different sets of four: eight
 * 32-column tiles per item.  The batch rows 32..63 of the A operand are the
 * weight rows of the same swizzle atom (batch <= 32 per pass): their products
 * land in accumulator rows that are never read, so both operands of a chunk fit
 * in 32 KB.
 *
 * Accumulators: TMEM columns [256 (i mod 2), 256 (i mod 2) + 256) for the i-th
 * item of the CTA.  One chunk into the next item (or at the end), the 8 warps of
 * each lane quarter that holds batch rows read 4 of the 32 columns each
 * (tcgen05.ld 32x32b) and add the eight tiles in a fixed order: with M = 64,
 * accumulator row 16 q + i sits in TMEM lane 32 q + i.  Row r of the item goes
 * to y[b][row0 + r]: stored, or added when a row spans tiles.
 */
constexpr int kMmaChunk = 256;                  /* columns per chunk */
constexpr uint32_t kMmaBufBytes = 32768u;       /* one chunk: 4 swizzle atoms of 8 KB */
constexpr uint32_t kMmaAtomBytes = 8192u;       /* 64 rows x 128 B: x rows 0..31, then weight rows 0..31 */
constexpr int kMmaMaxBatch = 32;                /* x rows per pass */
constexpr int kMmaMaxBufs = 3;                 /* chunk buffers in flight: 3 where shared memory allows, else 2 */
/* chunk buffers, barriers and the read slack after the last code pool */
__host__ __device__ constexpr size_t mma_fixed_bytes(int nbuf) { return (size_t)nbuf * kMmaBufBytes + 96 + kSlackBytes; }

__device__ __forceinline__ void sts128(uint32_t a, uint32_t x, uint32_t y, uint32_t z, uint32_t w) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(x), "r"(y), "r"(z), "r"(w) : "memory");
}
__device__ __forceinline__ void mbar_init_n(uint32_t mbar, uint32_t n) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(mbar), "r"(n) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t mbar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(mbar) : "memory");
}
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

/* Shared-memory matrix descriptor of a 128-byte-swizzled K-major operand whose
 * 8-row groups are 1024 bytes apart: start address >> 4 (bits 0..13), leading
 * offset 16 B (unused by swizzled K-major layouts), stride offset 1024 B >> 4
 * (bits 32..45), the descriptor version 1 (bit 46) and swizzle mode 2 = 128 B
 * (bits 61..63).  Stepping K by 16 inside a 64-column atom adds 32 bytes to the
 * start; the swizzle is applied to the absolute address, so atoms are 1024-aligned. */
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1u << 16) | ((uint64_t)(1024u >> 4) << 32) |
           ((uint64_t)1u << 46) | ((uint64_t)2u << 61);
}

/* One MMA, issued by one elected lane of a converged warp (the operands are warp-uniform). */
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
/* The completion of the elected lane's earlier MMAs arrives on mbar (converged warp). */
__device__ __forceinline__ void tc_commit(uint32_t mbar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(mbar)
        : "memory");
}

/* 2D tiled TMA load of one box (columns x0.., rows y0..) into shared memory,
 * completing on mbar (x0 is a multiple of 64 columns: 128-byte aligned). */
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int32_t x0, int32_t y0,
                                            uint32_t mbar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"((uint64_t)map), "r"(x0), "r"(y0), "r"(mbar)
        : "memory");
}

/* 32 lanes x 4 columns of 32 bits from TMEM (the lane quarter of the calling warp). */

/* The item a warp works on: matrix, first row, tile column, and the combined
 * index of the tile of the warp's row (have = the row exists). */
struct MmaItem {
    int mi;
    int64_t row0, tc, g;
    bool have;
};

__device__ __forceinline__ MmaItem mma_item(const HuffMmaArgs& a, int64_t it, int rows, int d) {
    MmaItem r;
    r.mi = 0;
    while (r.mi + 1 < a.count && it >= a.item_begin[r.mi + 1]) ++r.mi;
    const HuffMat& M = a.m[r.mi];
    const int64_t R = a.row_tiles[r.mi], local = it - a.item_begin[r.mi];
    const int64_t rb = local / R;
    r.tc = local - rb * R;
    r.row0 = rb * rows;
    const int64_t row = r.row0 + d;
    r.have = d >= 0 && d < rows && row < M.n_rows;
    r.g = M.tile_begin + (r.have ? row * R + r.tc : 0);
    return r;
}

__device__ __forceinline__ TileRef mma_tile(const HuffMmaArgs& a, const MmaItem& it) {
    if (it.have) return tile_ref(a, it.g, tile_offsets(a, it.g));
    TileRef r{};
    r.mi = it.mi;
    r.S = a.m[it.mi].steps;
    return r; /* area 0: nothing to copy or decode */
}

/* What the readout of a finished item needs. */
struct MmaDone {
    int mi;
    int64_t row0;
    uint32_t dcol;  /* its accumulator tiles */
    uint32_t s, ph; /* buffer and phase parity of its last chunk */
};

template <bool kHier>
__global__ void __launch_bounds__(kMaxHW * 32, 1) huff_mma_kernel(const __grid_constant__ HuffMmaArgs a) {
    extern __shared__ __align__(1024) uint8_t mma_smem[]; /* (the dynamic block, 1 KB aligned) */
    uint8_t* const smem = mma_smem;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarp = blockDim.x >> 5;
    const int rows = nwarp - 1, d = warp - 1; /* warp 0 produces; warps 1.. decode rows 0.. of the item */
    if (smem_u32(smem) & 1023u) { /* the swizzled operands need 1 KB alignment (never seen otherwise) */
        if (threadIdx.x == 0) flag_corrupt(a.status);
        return;
    }
    /* shared: nbuf chunk buffers | pair tables | staged sub-tables | two code pools
     * (items alternate) | the pools' mbarriers | full, done, xfull [nbuf each] | TMEM
     * address | slack.  A lane's reads run up to kSlackBytes past its tile's code area:
     * into the next tile, the other pool, the mbarriers or the slack, all inside the
     * block. */
    const uint32_t ops = smem_u32(smem);
    const int nbuf = a.nbuf;
    const uint32_t tabs_s = ops + (uint32_t)nbuf * kMmaBufBytes;
    uint32_t* const subs = (uint32_t*)(smem + (size_t)nbuf * kMmaBufBytes + (size_t)a.count * kPairTabBytes);
    const uint32_t pools = tabs_s + (uint32_t)a.count * kPairTabBytes + 4u * (uint32_t)a.sub_words;
    const uint32_t mbars = pools + 2u * (uint32_t)a.pool_bytes; /* pool p complete: all decoding warps' copies */
    const uint32_t full = mbars + 16, done = full + 24, xfull = full + 48, tslot = full + 72;
    const int64_t n_items = a.item_begin[a.count];

    /* A decoding warp's tile of an item goes into pool p, packed after the tiles of
     * the item's earlier rows (64 bytes of lane starts + the code area each, sizes
     * from the tile offsets, a prefix sum over the lanes); `region` receives its
     * place.  A tile that does not fit (corrupt offsets only) comes back with area 0. */
    auto stage = [&](const MmaItem& itm, uint32_t p, uint32_t& region) -> TileRef {
        const HuffMat& M = a.m[itm.mi];
        const int64_t row = itm.row0 + lane;
        uint32_t sz = 0;
        if (lane < rows && row < M.n_rows) {
            const int64_t g = M.tile_begin + row * a.row_tiles[itm.mi] + itm.tc;
            const TileRef r = tile_ref(a, g, tile_offsets(a, g));
            sz = r.area > 0 ? 64u + (uint32_t)r.area : 0u;
        }
        uint32_t inc = sz;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t v = __shfl_up_sync(kFull, inc, o);
            if (lane >= o) inc += v;
        }
        const uint32_t off = __shfl_sync(kFull, inc - sz, d);
        TileRef r = mma_tile(a, itm);
        if (r.area > 0 && off + 64u + (uint32_t)r.area > (uint32_t)a.pool_bytes) r.area = 0;
        region = pools + p * (uint32_t)a.pool_bytes + off;
        prefetch_code(region, mbars + 8 * p, r, lane, r.area);
        return r;
    };

    if (lane == 0) {
        if (d < 0) {
            mbar_init_n(mbars, (uint32_t)rows);
            mbar_init_n(mbars + 8, (uint32_t)rows);
            for (int i = 0; i < nbuf; ++i) {
                mbar_init_n(full + 8 * i, (uint32_t)rows);
                mbar_init(done + 8 * i);
                mbar_init(xfull + 8 * i);
            }
        }
        mbar_fence_init();
    }
    __syncthreads(); /* the pools' mbarriers (set up by warp 0) before any copy arrives on them */
    int64_t it = blockIdx.x;
    MmaItem ci = mma_item(a, it, rows, d);
    TileRef cur{};
    uint32_t region = 0; /* this warp's tile in the current pool */
    bool fits = true;    /* the next item's tile found room */
    if (d >= 0) cur = stage(ci, 0, region);
    for (int k = 0; k < a.count; ++k)
        stage_pair_table((uint32_t*)(smem + (tabs_s - smem_u32(smem)) + (size_t)k * kPairTabBytes), a.m[k].table);
    if (kHier) stage_sub_tables(a, subs);
    if (warp == 0) { /* all 512 TMEM columns: 2 items x 8 accumulator tiles of 32 columns */
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(tslot) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    grid_dep_launch();
    grid_dep_wait(); /* x and y belong to the preceding kernel in the stream from here on */
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = lds32(tslot);

    /* bounded waits; after one runs out (never seen: it needs a lost arrival) the
     * thread stops waiting, so a fault in the pipeline cannot hold the SM for long */
    bool live = true;
    auto wait = [&](uint32_t bar, uint32_t parity) {
        if (live && !mbar_wait(bar, parity)) {
            live = false;
            flag_corrupt(a.status);
        }
        return live;
    };
    /* x of a chunk (its columns from col on) into buffer s: 4 boxes of 32 rows x 64 columns */
    auto load_x = [&](uint32_t s, uint32_t col) {
        const uint32_t b = ops + s * kMmaBufBytes, bar = xfull + 8 * s;
        mbar_arrive_tx(bar, 4u * 32u * 128u);
#pragma unroll
        for (int at = 0; at < 4; ++at) tma_load_2d(b + at * kMmaAtomBytes, &a.xmap, (int32_t)(col + 64 * at), 0, bar);
    };
    /* y of a finished item: the warps of lane quarter q < 2 (batch rows 16 q ..) take 4
     * of its 32 columns each and add the 8 partial tiles in a fixed order */
    auto readout = [&](const MmaDone& f) {
        const int q = warp & 3, j = warp >> 2;
        if (q >= 2 || 16 * q >= a.batch || 4 * j >= rows) return;
        /* one lane issues every MMA and a commit covers all of that lane's earlier ones, so
         * the last chunk's suffices; no later chunk on its barrier can have completed yet
         * (the next one on it needs this warp's stores, or, for the producer, its issue) */
        wait(done + 8 * f.s, f.ph);
        tc_fence_after();
        float s[4] = {0.f, 0.f, 0.f, 0.f};
        const uint32_t t0 = tmem + ((uint32_t)(32 * q) << 16) + f.dcol + 4u * j;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t v[4][4];
#pragma unroll
            for (int t = 0; t < 4; ++t) tc_ld4(t0 + 32u * (4 * h + t), v[t]);
            tc_wait_ld();
#pragma unroll
            for (int t = 0; t < 4; ++t)
#pragma unroll
                for (int c = 0; c < 4; ++c) s[c] += __uint_as_float(v[t][c]);
        }
        tc_fence_before();
        const HuffMat& M = a.m[f.mi];
        const int b = 16 * q + lane;
        if (lane < 16 && b < a.batch) {
            float* yb = M.y + (int64_t)b * M.n_rows + f.row0;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int r = 4 * j + c;
                if (r < rows && f.row0 + r < M.n_rows) {
                    if (M.atomic_y) atomicAdd(yb + r, s[c]);
                    else yb[r] = s[c];
                }
            }
        }
    };

    uint32_t gc = 0;  /* chunks of this CTA so far */
    MmaDone prev{};
    bool have_prev = false;
    /* chunk gc sits in buffer bs = gc % nbuf; bp = (gc / nbuf) & 1 is the parity of that use
     * of the buffer's mbarriers (the previous use of the buffer had bp ^ 1) */
    uint32_t bs = 0, bp = 0;
    auto advance = [&]() {
        ++gc;
        if (++bs == (uint32_t)nbuf) {
            bs = 0;
            bp ^= 1u;
        }
    };
    if (d < 0 && lane == 0) { /* x of the first nbuf - 1 chunks (an item has at least 2) */
        const uint32_t col0 = (uint32_t)(ci.tc * 32 * a.m[ci.mi].steps);
        for (int j = 0; j + 1 < nbuf; ++j) load_x((uint32_t)j, col0 + (uint32_t)j * kMmaChunk);
    }
    for (uint32_t iter = 0; it < n_items; it += gridDim.x, ++iter) {
        const HuffMat& M = a.m[ci.mi];
        const int nch = M.steps / 8;
        const uint32_t dcol = 256u * (iter & 1u); /* this item's 8 accumulator tiles */
        const uint32_t col_t = (uint32_t)ci.tc * 32u * (uint32_t)M.steps;
        const int64_t nit = it + gridDim.x;
        if (d < 0) {
            /* ---- producer: x one chunk ahead, then the chunk's 16 MMAs ---- */
            for (int ch = 0; ch < nch; ++ch, advance()) {
                const uint32_t opb = ops + bs * kMmaBufBytes;
                /* the whole warp runs this loop (its values stay warp-uniform); one lane
                 * starts the copies, one elected lane issues each MMA */
                wait(full + 8 * bs, bp);
                wait(xfull + 8 * bs, bp);
                tc_fence_after();
                /* accumulator tile 4 (chunk & 1) + (k step & 3): four independent chains per
                 * chunk, consecutive chunks on different tiles */
                const uint32_t dt = tmem + dcol + 128u * (uint32_t)(ch & 1);
                const uint64_t ad = sw128_desc(opb), bd = sw128_desc(opb + 4096u);
#pragma unroll
                for (int ks = 0; ks < kMmaChunk / 16; ++ks) {
                    const uint64_t off = (uint64_t)(((ks >> 2) * kMmaAtomBytes + (ks & 3) * 32) >> 4);
                    tc_mma_bf16(dt + 32u * (ks & 3), ad + off, bd + off, a.idesc, ch > 1 || ks > 3);
                }
                tc_commit(done + 8 * bs);
                /* x of chunk gc + nbuf - 1, into the buffer of chunk gc - 1 once its MMAs are done */
                const int ahead = ch + nbuf - 1; /* in this item's numbering; the next item follows */
                if (ahead < nch || nit < n_items) {
                    uint32_t xcol;
                    if (ahead < nch) {
                        xcol = col_t + (uint32_t)ahead * kMmaChunk;
                    } else {
                        const MmaItem ni = mma_item(a, nit, rows, d);
                        xcol = (uint32_t)ni.tc * 32u * (uint32_t)a.m[ni.mi].steps + (uint32_t)(ahead - nch) * kMmaChunk;
                    }
                    const uint32_t ps = bs == 0 ? (uint32_t)nbuf - 1 : bs - 1, pp = bs == 0 ? bp ^ 1u : bp;
                    if (gc >= 1) wait(done + 8 * ps, pp);
                    if (lane == 0) load_x(ps, xcol);
                }
                __syncwarp();
                if (ch == 0 && have_prev) readout(prev); /* the previous item, one chunk late */
            }
        } else {
            /* ---- decoders: 8 symbols of the warp's row per chunk ---- */
            const uint32_t pi = iter & 1u;
            const bool arrived = wait(mbars + 8 * pi, (iter >> 1) & 1u); /* this item's tile */
            __syncwarp();
            if (!arrived) cur.area = 0;
            const uint32_t cb = region;
            if (nit < n_items) {
                /* the other pool held the previous item: every decoding warp is done with it
                 * once all have stored that item's last chunk.  (The next item's tile is
                 * resolved again at the end; only whether it fit is kept.) */
                if (have_prev) wait(full + 8 * prev.s, prev.ph);
                fits = stage(mma_item(a, nit, rows, d), pi ^ 1u, region).area > 0 || !mma_item(a, nit, rows, d).have;
            }
            /* the staged tile: lane starts, code area, window records (all of them: the pools
             * are sized for whole tiles) */
            const TileRecs tr = ci.have ? tile_recs(cb, cur.area, cur.area) : TileRecs{-1, 0u, 0u};
            if (ci.have && tr.n < 0 && lane == 0) flag_corrupt(a.status);
            const bool dec = tr.n >= 0;
            const uint32_t cbytes = tr.code;
            const uint32_t tab = tabs_s + (uint32_t)ci.mi * kPairTabBytes, area = cb + 64;
            const HierCtx hc = hier_ctx(a.m[ci.mi], subs, a.status);
            const uint32_t limit = area + cbytes;
            Lane s{};
            uint32_t s1 = 0;
            uint4 rr[2] = {};
            const uint4* raw4 = (const uint4*)(cur.rec + 64) + lane;
            uint2 rc = make_uint2(0u, 0u); /* the tile's window records: (applied, count) */
            if (dec) {
                const uint32_t s0 = lane ? lds16(cb + 2 * lane) : 0u;
                s1 = lane < 31 ? lds16(cb + 2 * lane + 2) : 0u;
                lane_seek(s, area, 8u * min(s0, cbytes));
                rr[0] = __ldg(raw4);
                if (nch > 2) rr[1] = __ldg(raw4 + 32);
                rc = make_uint2(0u, (uint32_t)tr.n);
            }
            const uint32_t seg = (uint32_t)(lane >> 3) * kMmaAtomBytes + ((uint32_t)((lane & 7) ^ (d & 7)) << 4) +
                                 4096u + (uint32_t)d * 128u;
            auto chunk = [&](int ch, uint32_t r0, uint32_t r1) {
                uint32_t w[4] = {0u, 0u, 0u, 0u};
                if (dec) {
                    lane_clamp(s, limit);
                    decode8<kHier>(s, tab, hc, r0, r1, w);
                }
                /* the buffer is free once the MMAs of its previous chunk (gc - nbuf) are done */
                if (gc >= (uint32_t)nbuf) wait(done + 8 * bs, bp ^ 1u);
                const uint32_t opb = ops + bs * kMmaBufBytes;
                sts128(opb + seg, w[0], w[1], w[2], w[3]);
                /* window records of this chunk (tile positions below 256 (ch + 1)): the
                 * true weight over the coded one, at its lane's row segment */
                if (rc.x < rc.y) {
                    __syncwarp();
                    while (rc.x < rc.y) {
                        const uint32_t idx = rc.x + (uint32_t)lane;
                        const uint32_t e = idx < rc.y ? lds32(cb + 64 + cbytes + 4 * idx) : 0xFFFFFFFFu;
                        const uint32_t q = rec_pos(e);
                        const bool in = idx < rc.y && q < 256u * (uint32_t)(ch + 1);
                        if (in) {
                            const uint32_t lr = (q >> 3) & 31u;
                            const uint32_t at = opb + (lr >> 3) * kMmaAtomBytes + (((lr & 7u) ^ (uint32_t)(d & 7)) << 4) +
                                                4096u + (uint32_t)d * 128u + 2u * (q & 7u);
                            const uint32_t wt = rec_weight(e, rec_exp(e));
                            asm volatile("st.shared.u16 [%0], %1;" ::"r"(at), "h"((unsigned short)wt) : "memory");
                        }
                        const uint32_t n = (uint32_t)__popc(__ballot_sync(kFull, in));
                        rc.x += n;
                        if (n < 32) break;
                    }
                }
                fence_async_smem(); /* the tensor cores read what the generic stores wrote */
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(full + 8 * bs);
                advance();
            };
            const int nb = nch / 2; /* raw blocks of 16 symbols; block b + 2 is loaded once block b is decoded */
            for (int b0 = 0; b0 < nb; b0 += 2) {
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int blk = b0 + u;
                    if (u == 0 || blk < nb) {
                        chunk(2 * blk, rr[u].x, rr[u].y);
                        if (u == 0 && b0 == 0 && have_prev) readout(prev); /* the previous item, one chunk late */
                        chunk(2 * blk + 1, rr[u].z, rr[u].w);
                        if (dec && blk + 2 < nb) rr[u] = __ldg(raw4 + 32 * (blk + 2));
                    }
                }
            }
            /* every lane's codewords end in the last byte before the next lane's start */
            const uint32_t p = lane_pos(s, area), pmax = 8u * cbytes;
            const bool bad = dec && (lane < 31 ? (p > 8u * s1 || p + 8u <= 8u * s1) : (p + 64u > pmax));
            if (__any_sync(kFull, bad) && lane == 0) flag_corrupt(a.status);
        }
        prev.mi = ci.mi;
        prev.row0 = ci.row0;
        prev.dcol = dcol;
        prev.s = bs == 0 ? (uint32_t)nbuf - 1 : bs - 1; /* the item's last chunk, gc - 1 */
        prev.ph = bs == 0 ? bp ^ 1u : bp;
        have_prev = true;
        if (nit < n_items) {
            ci = mma_item(a, nit, rows, d);
            cur = mma_tile(a, ci);
            if (!fits) cur.area = 0;
        }
    }
    if (have_prev) readout(prev);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
    }
}

/* ============================================== tensor-core GEMM (prefill) */
/*
 * Batch > 1 materialises the layer and runs a GEMM (MINE, "Prefill"; DFloat11,
 * "Transformer-block-level decompression"): here the decoded rows arrive in an
 * L2-sized chunk of BF16 [rows, ld] and this kernel forms y[b][row] = sum_k
 * W[row][k] x[b][k] over it.
 *
 * Tile: 128 weight rows (MMA M, the TMEM lanes) x bn batch rows (MMA N, TMEM
 * columns, a multiple of 16 up to 256), K in blocks of 64 columns (one 128-byte
 * swizzle atom).  Per block a stage of shared memory holds the A box (128 rows x
 * 128 B) and the B box (bn rows x 128 B), both 128-byte swizzled by TMA; four
 * kind::f16 MMAs of K = 16 consume it.  Warp roles: warp 0 issues the TMA copies
 * (one lane), warp 1 the MMAs (one elected lane), warps 2..5 read the finished
 * accumulators back (tcgen05.ld 32x32b, lane quarter = warp % 4) and store them:
 * for a batch row b the 32 lanes of a warp hold 32 consecutive weight rows, so
 * each store is 128 contiguous bytes.  Two accumulators (2 bn TMEM columns)
 * alternate between work items so that the read-back of one overlaps the MMAs of
 * the next.  A work item is (row tile, batch tile, K split); with more than one K
 * split each writes its own partial sums, which gemm_reduce_kernel adds in split
 * order, so results do not depend on timing.
 *
 * Barriers: full[s] (TMA bytes landed), empty[s] (the MMAs that read stage s are
 * done: tcgen05.commit), accf[a] (accumulator a complete), acce[a] (its read-back
 * done: one arrival per epilogue warp).  Every wait is bounded; a wait that runs
 * out flags the status word and the thread stops waiting.
 */
constexpr int kGemmBM = 128;
constexpr int kGemmBK = 64;
constexpr int kGemmEpiWarps = 4;
constexpr int kGemmThreads = 32 * (2 + kGemmEpiWarps);
constexpr uint32_t kGemmABytes = (uint32_t)kGemmBM * 128u; /* 16 KB */

struct GemmArgs {
    CUtensorMap amap; /* W rows [rows, K] BF16, boxes of 64 columns x 128 rows, 128-byte swizzle */
    CUtensorMap bmap; /* x [batch, K] BF16, boxes of 64 columns x bn rows, 128-byte swizzle */
    float* y;         /* ksplit == 1: y[b * ldy + row_off + row] */
    float* part;      /* ksplit > 1: part[(split * batch + b) * rows + row] */
    int64_t ldy, row_off;
    int rows, batch, kblocks, bn;
    int m_tiles, n_tiles, ksplit, kb_per_split;
    int stages;
    uint32_t idesc;   /* kind::f16, M = 128, N = bn */
    uint32_t tmem_cols;
    int* status;
};

__device__ __forceinline__ void tc_ld16(uint32_t taddr, uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
          "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tc_wait_ld16(uint32_t (&v)[16]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]), "+r"(v[6]), "+r"(v[7]),
                   "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]), "+r"(v[12]), "+r"(v[13]), "+r"(v[14]),
                   "+r"(v[15])::"memory");
}

__global__ void __launch_bounds__(kGemmThreads, 1) gemm_bf16_kernel(const __grid_constant__ GemmArgs a) {
    extern __shared__ __align__(1024) uint8_t gemm_smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t base = smem_u32(gemm_smem);
    if (base & 1023u) { /* the swizzled operands need 1 KB alignment (never seen otherwise) */
        if (threadIdx.x == 0) flag_corrupt(a.status);
        return;
    }
    const uint32_t stage_bytes = kGemmABytes + (uint32_t)a.bn * 128u;
    const uint32_t bars = base + (uint32_t)a.stages * stage_bytes;
    const uint32_t full = bars, empty = bars + 8u * (uint32_t)a.stages, accf = empty + 8u * (uint32_t)a.stages,
                   acce = accf + 16u, tslot = acce + 16u;
    if (threadIdx.x == 0) {
        for (int s = 0; s < a.stages; ++s) {
            mbar_init(full + 8 * s);
            mbar_init(empty + 8 * s);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(accf + 8 * i);
            mbar_init_n(acce + 8 * i, kGemmEpiWarps);
        }
        mbar_fence_init();
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(tslot),
                     "r"(a.tmem_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = lds32(tslot);
    grid_dep_launch();
    grid_dep_wait(); /* the weight rows and x come from the preceding kernels in the stream */

    bool live = true;
    auto wait = [&](uint32_t bar, uint32_t parity) {
        if (live && !mbar_wait(bar, parity)) {
            live = false;
            flag_corrupt(a.status);
        }
        return live;
    };
    const int items = a.m_tiles * a.n_tiles * a.ksplit;
    auto item_of = [&](int it, int& mt, int& nt, int& kb0, int& kb1) {
        const int ks = it % a.ksplit, mn = it / a.ksplit;
        nt = mn % a.n_tiles;
        mt = mn / a.n_tiles;
        kb0 = ks * a.kb_per_split;
        kb1 = min(a.kblocks, kb0 + a.kb_per_split);
    };

    if (warp == 0) {
        /* ---- TMA producer ---- */
        if (lane == 0) {
            uint32_t s = 0, ph = 0;
            for (int it = blockIdx.x; it < items; it += gridDim.x) {
                int mt, nt, kb0, kb1;
                item_of(it, mt, nt, kb0, kb1);
                for (int kb = kb0; kb < kb1; ++kb) {
                    wait(empty + 8 * s, ph ^ 1u);
                    const uint32_t st = base + s * stage_bytes;
                    mbar_arrive_tx(full + 8 * s, stage_bytes);
                    tma_load_2d(st, &a.amap, kb * kGemmBK, mt * kGemmBM, full + 8 * s);
                    tma_load_2d(st + kGemmABytes, &a.bmap, kb * kGemmBK, nt * a.bn, full + 8 * s);
                    if (++s == (uint32_t)a.stages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
        }
    } else if (warp == 1) {
        /* ---- MMA issuer (the whole warp walks the loop; one elected lane issues) ---- */
        uint32_t s = 0, ph = 0, n = 0;
        for (int it = blockIdx.x; it < items; it += gridDim.x, ++n) {
            int mt, nt, kb0, kb1;
            item_of(it, mt, nt, kb0, kb1);
            const uint32_t ab = n & 1u, aph = (n >> 1) & 1u;
            wait(acce + 8 * ab, aph ^ 1u); /* the read-back of this accumulator's previous item is done */
            tc_fence_after();
            const uint32_t d = tmem + ab * (uint32_t)a.bn;
            for (int kb = kb0; kb < kb1; ++kb) {
                wait(full + 8 * s, ph);
                tc_fence_after();
                const uint32_t st = base + s * stage_bytes;
                const uint64_t ad = sw128_desc(st), bd = sw128_desc(st + kGemmABytes);
#pragma unroll
                for (int k = 0; k < kGemmBK / 16; ++k)
                    tc_mma_bf16(d, ad + (uint64_t)(2 * k), bd + (uint64_t)(2 * k), a.idesc, kb > kb0 || k > 0);
                tc_commit(empty + 8 * s);
                if (++s == (uint32_t)a.stages) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            tc_commit(accf + 8 * ab);
            __syncwarp();
        }
    } else {
        /* ---- epilogue: TMEM lanes 32 q .. 32 q + 31 = weight rows of the tile ---- */
        const int q = warp & 3;
        uint32_t n = 0;
        for (int it = blockIdx.x; it < items; it += gridDim.x, ++n) {
            int mt, nt, kb0, kb1;
            item_of(it, mt, nt, kb0, kb1);
            const uint32_t ab = n & 1u, aph = (n >> 1) & 1u;
            wait(accf + 8 * ab, aph);
            tc_fence_after();
            const int row = mt * kGemmBM + 32 * q + lane;
            const int ks = it % a.ksplit;
            const bool row_ok = row < a.rows;
            for (int c0 = 0; c0 < a.bn; c0 += 16) {
                uint32_t v[16];
                tc_ld16(tmem + ((uint32_t)(32 * q) << 16) + ab * (uint32_t)a.bn + (uint32_t)c0, v);
                tc_wait_ld16(v);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int b = nt * a.bn + c0 + j;
                    if (row_ok && b < a.batch) {
                        if (a.ksplit == 1) a.y[(int64_t)b * a.ldy + a.row_off + row] = __uint_as_float(v[j]);
                        else a.part[((int64_t)ks * a.batch + b) * a.rows + row] = __uint_as_float(v[j]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acce + 8 * ab);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(a.tmem_cols) : "memory");
    }
}

/* y[b * ldy + row_off + r] = sum over splits s (in order) of part[(s * batch + b) * rows + r]. */
__global__ void gemm_reduce_kernel(const float* __restrict__ part, int ksplit, int batch, int rows, float* y,
                                   int64_t ldy, int64_t row_off) {
    grid_dep_launch();
    grid_dep_wait();
    const int64_t n = (int64_t)batch * rows;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t b = i / rows, r = i - b * rows;
        float s = 0.f;
        for (int k = 0; k < ksplit; ++k) s += part[((int64_t)k * batch + b) * rows + r];
        y[b * ldy + row_off + r] = s;
    }
}

/* ---- not in the Huffman GEMV: end ---- */
/* ====================================================== Huffman decode kernel */
/* Each CTA owns a contiguous range of the launch's tiles; it walks the range one
 * matrix segment at a time, with that matrix's pair table in shared memory.
 * Every 8 symbols of a lane are 8 consecutive columns, so each lane stores them
 * with one 16-byte write and a warp writes 512 contiguous bytes. */


/* Window records of a decoded tile that starts at flattened position `start` of
 * its matrix: the true weight over the coded one (inline: most tiles have a few,
 * and a call would spill the walker's registers around it). */
__device__ __forceinline__ void decode_records(uint32_t recs, uint32_t staged, const uint32_t* far, uint32_t nrec,
                                            const HuffMat& M, int64_t start, int lane) {
    for (uint32_t j = (uint32_t)lane; j < nrec; j += 32) {
        const uint32_t e = j < staged ? lds32(recs + 4 * j) : __ldg(far + j), q = rec_pos(e);
        const int64_t f = start + q, rr = f / M.k_pad, cc = f - rr * M.k_pad;
        if (cc < M.k_cols) M.out[(rr - M.out_row0) * M.out_ld + cc] = (uint16_t)rec_weight(e, rec_exp(e));
    }
}

/* warps per CTA of the decode kernel (64 registers a thread) */
constexpr int kDecodeWarps = 32;

template <bool kHier>
__global__ void __launch_bounds__(kDecodeWarps * 32, 1) huff_decode_kernel(const __grid_constant__ HuffDecodeArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarp = blockDim.x >> 5;
    /* shared: the current matrix's pair table | its staged sub-tables | per warp: two tile buffers */
    uint4* tab = (uint4*)smem;
    uint32_t* subs = (uint32_t*)(smem + kPairTabBytes);
    uint8_t* wbase = smem + kPairTabBytes + 4 * (size_t)a.sub_words + (size_t)warp * huff_warp_bytes(a.code_bytes);
    const uint32_t bufs = smem_u32(wbase), buf_bytes = (uint32_t)tile_buf_bytes(a.code_bytes);
    const uint32_t tab_s = smem_u32(tab);
    const uint32_t mbars = bufs + 2 * buf_bytes;
    if (lane == 0) {
        mbar_init(mbars);
        mbar_init(mbars + 8);
        mbar_fence_init();
    }
    __syncwarp();
    uint32_t ph = 0; /* parity of the next phase of each buffer's mbarrier */
    grid_dep_launch();
    grid_dep_wait();

    const int64_t lo = a.total_tiles * blockIdx.x / gridDim.x, hi = a.total_tiles * (blockIdx.x + 1) / gridDim.x;
    for (int64_t cur = lo; cur < hi;) {
        const int mi = owner(a, cur);
        const HuffMat& M = a.m[mi];
        const int64_t mend = min(hi, M.tile_begin + M.n_tiles);
        const int64_t g0 = cur + warp;
        TileRef first{};
        if (g0 < mend) {
            first = tile_ref(a, g0, tile_offsets(a, g0));
            prefetch_code(bufs, mbars, first, lane, a.code_bytes);
        }
        __syncthreads();
        stage_pair_table((uint32_t*)tab, M.table);
        /* this matrix's sub-tables, when they were sized to fit (sub_smem == 0) */
        HuffMat Ms = M;
        if (kHier && M.sub_smem >= 0 && 256 * M.n_sub <= a.sub_words) {
            Ms.sub_smem = 0;
            const uint4* ss = (const uint4*)(M.table + EC_PAIR_WORDS);
            for (int i = threadIdx.x; i < 64 * M.n_sub; i += blockDim.x) ((uint4*)subs)[i] = __ldg(ss + i);
        } else {
            Ms.sub_smem = -1;
        }
        __syncthreads();
        const int64_t kp = M.k_pad, K = M.k_cols, ld = M.out_ld;
        /* 16-byte stores when rows are 16-byte aligned (a store past column K stays
         * inside the row: ld >= K rounded up to 8) */
        const bool vec = (ld % 8) == 0;
        /* the current row's output (lane-private: this lane's first column of the row's
         * segment) and the segment's first column; rows and columns stay below 2^31 */
        uint16_t* dst = nullptr;
        uint32_t col0 = 0;
        const uint32_t kp32 = (uint32_t)kp, K32 = (uint32_t)K;
        if (g0 < mend)
            huff_walk<kHier>(
                a, g0, nwarp, mend, first, bufs, buf_bytes, ph, lane,
                [&](int) {
                    WalkCtx c;
                    c.tab = tab_s;
                    c.h = hier_ctx(Ms, subs, a.status);
                    return c;
                },
                [&](const TileRef& r) {
                    const int64_t T = 32 * (int64_t)M.steps;
                    const int64_t row = tile_row(r.t, T, kp, EC_HUFF_ROW_ALIGN);
                    col0 = (uint32_t)(r.t * T - row * kp);
                    dst = M.out + (row - M.out_row0) * ld + 8 * lane;
                },
                [&](uint32_t, const TileRef&) {
                    if (col0 >= kp32) {
                        col0 -= kp32;
                        dst += ld;
                    }
                },
                [&](const uint32_t (&w)[4], int) {
                    /* the lane's 8 outputs are columns col0 + 8 lane .. + 7: one 16-byte store */
                    const uint32_t col = col0 + 8u * (uint32_t)lane;
                    if (vec) {
                        if (col < K32) *(uint4*)(dst + col0) = make_uint4(w[0], w[1], w[2], w[3]);
                    } else {
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            if (col + j < K32) dst[col0 + j] = (uint16_t)(w[j >> 1] >> (16 * (j & 1)));
                    }
                    col0 += 256;
                },
                [&](const TileRef& r, uint32_t cb, const TileRecs& tr) {
                    /* window records: the true weight over the coded one (stored above by
                     * some lane of this warp) */
                    if (tr.n > 0) {
                        __syncwarp();
                        decode_records(cb + 64 + tr.code, tr.staged, far_records(r, tr.code), (uint32_t)tr.n, M,
                                       32 * (int64_t)M.steps * r.t, lane);
                    }
                });
        cur = mend;
    }
}

/* ---- not in the Huffman GEMV: begin ---- */
/* x [batch, K] into shared rows of k_pad entries in the per-128-column permuted
 * order above (zero past K). */
__device__ __forceinline__ void stage_x_perm(uint16_t* xs, const uint16_t* __restrict__ x, int batch, int64_t K,
                                             uint32_t kp) {
    const uint32_t n = (uint32_t)batch * kp;
    for (uint32_t i = threadIdx.x; i < n; i += blockDim.x) {
        const uint32_t b = i / kp, q = i - b * kp, blk = q & ~127u, r = q & 127u;
        const uint32_t c = blk + 32u * (r & 3u) + (r >> 2);
        xs[i] = c < (uint32_t)K ? __ldg(x + (int64_t)b * K + c) : (uint16_t)0;
    }
}

/* x'-index of column c (the permutation above). */
__device__ __forceinline__ uint32_t x_perm_index(uint32_t c) { return (c & ~127u) + 4u * (c & 31u) + ((c >> 5) & 3u); }

/* The FP32 value of 4-bit symbol s (bits 0..3): the integer s - 8, or with fp4 the
 * FP4 E2M1 pattern s: bit 3 the sign, bits 1..2 the exponent field e (bias 1), bit
 * 0 the mantissa m; e = 0 gives m * 0.5, otherwise (1 + m / 2) * 2^(e - 1), i.e. the
 * FP32 pattern with biased exponent 126 + e and mantissa m << 22. */
__device__ __forceinline__ float code_value(uint32_t s, bool fp4) {
    if (!fp4) return __int_as_float(0x4B000000 | s) - 8388616.0f; /* (2^23 + s) - (2^23 + 8) */
    const uint32_t e = (s >> 1) & 3u, m = s & 1u;
    const uint32_t mag = e ? ((126u + e) << 23) | (m << 22) : (m ? 0x3F000000u : 0u);
    return __uint_as_float(mag | ((s & 8u) << 28));
}

/* ============================================================ rANS kernels */
/*
 * One warp per 4096-symbol tile (EntroPack, independent rANS tiles): lane l holds
 * state x_l and decodes positions 32 j + l.  A step looks the slot x & (2^b - 1)
 * up in the shared slot table (symbol, freq, slot - cum), sets
 * x = freq * (x >> b) + slot - cum, and lanes whose state fell below 2^16 pull the
 * next 16-bit word, in lane order (ballot + popc).  Words and the 32 initial
 * states of the warp's next tile arrive by cp.async into the second of two
 * shared buffers while the current tile is decoded.  Rows are multiples of 128
 * columns, so the scale group (128 consecutive weights, FP16) of 4 steps is one
 * value for the warp, and the scales of a tile's groups are contiguous: lane g
 * loads group g's scale at the start of the previous tile.  GEMV: sum code * x
 * over a group in FP32, then multiply by the group's scale (both exact up to the
 * FP32 sums); decode: BF16 round-to-nearest-even of code * scale (exact in FP32).
 */
__host__ __device__ constexpr int rans_max_warps(int b) { return b <= 1 ? 32 : (b <= 4 ? 24 : 16); }

/* one tile buffer: 32 states, the words (capacity rounded to 16 bytes), slack */
__host__ __device__ constexpr size_t rans_buf_bytes(int words_cap) {
    return 128 + (((size_t)words_cap * 2 + 15) & ~(size_t)15) + 64;
}

struct RansTile {
    const uint8_t* rec;
    int64_t t;
    int S;      /* symbols per lane */
    int words;  /* payload words; -1 = corrupt record (skipped) */
};

template <class Mat>
__device__ __forceinline__ RansTile rans_tile(const Mat& M, int64_t t, uint2 off) {
    RansTile r;
    r.t = t;
    r.S = t == M.n_tiles - 1 ? M.last_steps : M.steps;
    const int wb = (int)((off.y - off.x) * 16u) - 128;
    const bool ok = off.x <= off.y && off.y <= M.rec16 && wb >= 0 && wb <= 2 * M.words_cap;
    r.rec = M.records + (size_t)(ok ? off.x : 0u) * 16;
    r.words = ok ? wb / 2 : -1;
    return r;
}

__device__ __forceinline__ void rans_prefetch(uint32_t buf, const RansTile& r, int lane) {
    if (r.words >= 0) {
        if (lane < 8) cp_async16(buf + 16 * lane, r.rec + 16 * lane);
        for (int i = lane; i < r.words / 8; i += 32) cp_async16(buf + 128 + 16 * i, r.rec + 128 + 16 * i);
    }
    cp_async_commit();
}

__device__ __forceinline__ uint32_t lds16_if(bool p, uint32_t a, uint32_t v) {
    asm volatile("{\n\t.reg .pred q;\n\t.reg .b16 h;\n\t"
                 "setp.ne.u32 q, %1, 0;\n\t"
                 "@q ld.shared.u16 h, [%2];\n\t"
                 "@q cvt.u32.u16 %0, h;\n\t}"
                 : "+r"(v)
                 : "r"((uint32_t)p), "r"(a)
                 : "memory");
    return v;
}

template <bool kGemv, int B, bool kPair>
__global__ void __launch_bounds__(rans_max_warps(B) * 32, 1) rans_kernel(const __grid_constant__ RansArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    const RansMat& M = a.m;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarp = blockDim.x >> 5;
    const uint32_t kp = (uint32_t)M.k_pad;
    const int64_t K = M.k_cols;
    const int pb = M.prob_bits;
    const uint32_t mask_b = (1u << pb) - 1;
    const int batch = kGemv ? a.batch : 0;
    /* shared: slot table | (GEMV) 256 code pairs as packed BF16 | (GEMV) x, permuted per
     * 128 columns | two tile buffers per warp */
    const uint32_t tab_s = smem_u32(smem), lut_s = tab_s + (4u << pb);
    uint16_t* xs = (uint16_t*)(smem + ((size_t)4 << pb) + (kGemv ? 1024 : 0));
    const uint32_t xs_s = smem_u32(xs);
    const uint32_t buf_bytes = (uint32_t)rans_buf_bytes(M.words_cap);
    const uint32_t bufs = xs_s + (uint32_t)(2 * (size_t)batch * kp) + (uint32_t)warp * 2 * buf_bytes;
    const uint32_t cap = (buf_bytes - 128) / 2 - 1; /* last word index inside the buffer */
    const int64_t T = 32 * (int64_t)M.steps;

    const int64_t gw = (int64_t)blockIdx.x * nwarp + warp, nw = (int64_t)gridDim.x * nwarp;
    RansTile cur{};
    float sc = 0.f; /* lane g: scale of group g of the current tile */
    if (kGemv) /* entry i: [bf16(v1) | bf16(v0)], v0 the value of symbol i >> 4 (the earlier step), v1 of i & 15 */
        for (int i = threadIdx.x; i < 256; i += blockDim.x) {
            const bool fp4 = M.values == EC_RANS_VALUES_FP4_E2M1;
            const uint32_t c0 = __bfloat16_as_ushort(__float2bfloat16_rn(code_value((uint32_t)i >> 4, fp4)));
            const uint32_t c1 = __bfloat16_as_ushort(__float2bfloat16_rn(code_value((uint32_t)i & 15u, fp4)));
            asm volatile("st.shared.u32 [%0], %1;" ::"r"(lut_s + 4u * (uint32_t)i), "r"(c0 | (c1 << 16)) : "memory");
        }
    if (gw < M.n_tiles) {
        cur = rans_tile(M, gw, make_uint2(__ldg(M.tile_off + gw), __ldg(M.tile_off + gw + 1)));
        rans_prefetch(bufs, cur, lane);
        const int64_t g0 = gw * (T / 128) + lane;
        if (lane < cur.S / 4) sc = __half2float(__ushort_as_half(__ldg(M.scales + g0)));
    }
    {
        const uint4* src = (const uint4*)M.table;
        uint4* dst = (uint4*)smem;
        for (int i = threadIdx.x; i < (1 << pb) / 4; i += blockDim.x) dst[i] = __ldg(src + i);
    }
    grid_dep_launch();
    grid_dep_wait(); /* x, y and out belong to the preceding kernel in the stream from here on */
    if (kGemv) stage_x_perm(xs, a.x, batch, K, kp);
    __syncthreads();
    if (gw >= M.n_tiles) return;

    uint2 off_next = gw + nw < M.n_tiles ? make_uint2(__ldg(M.tile_off + gw + nw), __ldg(M.tile_off + gw + nw + 1))
                                         : make_uint2(0u, 0u);
    const uint32_t lt = (1u << lane) - 1u;
    uint32_t cb = bufs;
    for (int64_t t = gw; t < M.n_tiles; t += nw) {
        cp_async_wait_all();
        __syncwarp();
        const uint32_t nb_buf = cb == bufs ? bufs + buf_bytes : bufs;
        RansTile nxt{};
        float sc_next = 0.f;
        if (t + nw < M.n_tiles) {
            nxt = rans_tile(M, t + nw, off_next);
            rans_prefetch(nb_buf, nxt, lane);
            if (lane < nxt.S / 4) sc_next = __half2float(__ushort_as_half(__ldg(M.scales + (t + nw) * (T / 128) + lane)));
            if (t + 2 * nw < M.n_tiles)
                off_next = make_uint2(__ldg(M.tile_off + t + 2 * nw), __ldg(M.tile_off + t + 2 * nw + 1));
        }
        if (cur.words < 0) {
            if (lane == 0) flag_corrupt(a.status);
        } else {
            uint32_t x = lds32(cb + 4 * lane);
            const uint32_t wbase = cb + 128;
            uint32_t wp = 0;
            int64_t row = tile_row(t, T, kp, EC_RANS_ROW_ALIGN);
            uint32_t col = (uint32_t)(t * T - row * (int64_t)kp) + lane; /* this lane's column */
            float acc[B];
#pragma unroll
            for (int b = 0; b < B; ++b) acc[b] = 0.f;
            auto flush = [&]() {
#pragma unroll
                for (int b = 0; b < B; ++b) {
                    if (B > 1 && b >= batch) break;
                    const float v = warp_sum(acc[b]);
                    if (lane == 0) {
                        float* dst = M.y + (int64_t)b * M.n_rows + row;
                        if (M.atomic_y) atomicAdd(dst, v);
                        else *dst = v;
                    }
                    acc[b] = 0.f;
                }
            };
            const int ng = cur.S / 4;
            for (int gi = 0; gi < ng; ++gi) {
                if (col >= kp) { /* rows start on group boundaries */
                    if (kGemv) flush();
                    col -= kp;
                    ++row;
                }
                if ((gi & 31) == 0 && gi > 0) /* tiles of more than 32 groups */
                    sc = lane < ng - gi ? __half2float(__ushort_as_half(__ldg(M.scales + t * (T / 128) + gi + lane)))
                                        : 0.f;
                const float scale = __shfl_sync(kFull, sc, gi & 31);
                if (kGemv) {
                    /* one rANS step: the slot entry of the decoded symbol */
                    auto step = [&]() {
                        const uint32_t e = lds32(tab_s + ((x & mask_b) << 2));
                        if (kPair) { /* freq - 1 in bits 20..31: f X = (f - 1) X + X */
                            const uint32_t X = x >> pb;
                            x = (e >> 20) * X + X + ((e >> 8) & 0xFFFu);
                        } else {
                            x = (e >> 16) * (x >> pb) + ((e >> 4) & 0xFFFu);
                        }
                        const bool need = x < 65536u;
                        const uint32_t bal = __ballot_sync(kFull, need);
                        const uint32_t idx = min(wp + __popc(bal & lt), cap);
                        const uint32_t v = lds16_if(need, wbase + 2 * idx, 0u);
                        x = need ? x * 65536u + v : x;
                        wp += __popc(bal);
                        return e;
                    };
                    /* the group's four codes (lane steps 4 gi .. 4 gi + 3, columns col + 32 k) as
                     * two packed BF16 pairs from the code-pair table: a pair symbol's earlier
                     * code sits in bits 4..7, a single code in bits 0..3 */
                    uint32_t w01, w23;
                    if (kPair) {
                        w01 = lds32(lut_s + ((step() & 0xFFu) << 2));
                        w23 = lds32(lut_s + ((step() & 0xFFu) << 2));
                    } else {
                        const uint32_t e0 = step() & 15u, e1 = step() & 15u, e2 = step() & 15u, e3 = step() & 15u;
                        w01 = lds32(lut_s + (((e0 << 4) | e1) << 2));
                        w23 = lds32(lut_s + (((e2 << 4) | e3) << 2));
                    }
                    /* x of the four columns, one 8-byte load per batch row (permuted layout);
                     * the exact products are summed in FP32, then scaled by the group's scale */
                    const uint32_t xa = xs_s + 2u * ((col - (uint32_t)lane) + 4u * (uint32_t)lane);
#pragma unroll
                    for (int b = 0; b < B; ++b) {
                        if (B > 1 && b >= batch) break;
                        uint2 xq;
                        asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(xq.x), "=r"(xq.y) : "r"(xa + 2u * (uint32_t)b * kp));
                        float g0 = 0.f, g1 = 0.f;
                        fma2x_bf16(w01, xq.x, g0, g1);
                        fma2x_bf16(w23, xq.y, g0, g1);
                        acc[b] = fmaf(g0 + g1, scale, acc[b]);
                    }
                    col += 128;
                    continue;
                }
#pragma unroll
                for (int s = 0; s < (kPair ? 2 : 4); ++s) {
                    const uint32_t e = lds32(tab_s + ((x & mask_b) << 2));
                    if (kPair) { /* freq - 1 in bits 20..31: f X = (f - 1) X + X */
                        const uint32_t X = x >> pb;
                        x = (e >> 20) * X + X + ((e >> 8) & 0xFFFu);
                    } else {
                        x = (e >> 16) * (x >> pb) + ((e >> 4) & 0xFFFu);
                    }
                    const bool need = x < 65536u;
                    const uint32_t bal = __ballot_sync(kFull, need);
                    const uint32_t idx = min(wp + __popc(bal & lt), cap);
                    const uint32_t v = lds16_if(need, wbase + 2 * idx, 0u);
                    x = need ? x * 65536u + v : x; /* v < 2^16 and x < 2^16: the shift-or as one multiply-add */
                    wp += __popc(bal);
                    /* a symbol in the low 4 bits (pairs: the lane's earlier step in bits 4..7, the
                     * later one in bits 0..3), its value exact in FP32 */
                    const int nc = kPair ? 2 : 1;
#pragma unroll
                    for (int q = 0; q < nc; ++q) {
                        const uint32_t nib = kPair ? (q == 0 ? (e >> 4) & 15u : e & 15u) : e & 15u;
                        const float cf = code_value(nib, M.values == EC_RANS_VALUES_FP4_E2M1);
                        const uint32_t c = col + 32 * (nc * s + q);
                        if (c < K) M.out[row * K + c] = __bfloat16_as_ushort(__float2bfloat16_rn(cf * scale));
                    }
                }
                col += 128;
            }
            /* every lane returns to its initial state 2^16 and the words are used up
             * (the encoder pads the words to 16 bytes: up to 7 trailing zeros) */
            if (__any_sync(kFull, x != 65536u) || wp > (uint32_t)cur.words || (uint32_t)cur.words - wp > 7) {
                if (lane == 0) flag_corrupt(a.status);
            }
            if (kGemv) flush();
        }
        cur = nxt;
        sc = sc_next;
        cb = nb_buf;
    }
}

/* ============================================================== FP8 kernel */
/* FP8 weights under a top-t table (MINE section 4, "Escapes"): the rANS tiles
 * decode one table symbol per position (pair-layout slot entries: symbol, slot
 * bias, frequency - 1), the symbol's FP32 value feeds the FMA (GEMV) or is scaled
 * by the row scale and stored (decode); a weight outside the table was coded as
 * code 0 (value 0).  GEMV: before each row's warp reduction the lanes take that
 * row's correction records in turn and add value * x to their own sums (the row
 * scale then multiplies the whole sum), so no record needs an atomic of its own;
 * decode: after its tile the warp writes bf16(value * r_i) over the 0. */
template <bool kGemv, int B>
__global__ void __launch_bounds__(rans_max_warps(B) * 32, 1) fp8_kernel(const __grid_constant__ Fp8Args a) {
    extern __shared__ __align__(16) uint8_t smem[];
    const Fp8Mat& M = a.m;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarp = blockDim.x >> 5;
    const uint32_t kp = (uint32_t)M.k_pad;
    const int64_t K = M.k_cols;
    const int pb = M.prob_bits;
    const uint32_t mask_b = (1u << pb) - 1;
    const int batch = kGemv ? a.batch : 0;
    const uint32_t tab_s = smem_u32(smem);
    const size_t tab_bytes = ((size_t)4 << pb) + 4 * EC_FP8_VALUE_WORDS;
    const float* vals = (const float*)(smem + ((size_t)4 << pb)); /* [0, 256): symbols, [256, 512): codes */
    uint16_t* xs = (uint16_t*)(smem + tab_bytes);
    const uint32_t buf_bytes = (uint32_t)rans_buf_bytes(M.words_cap);
    const uint32_t bufs = smem_u32(xs) + (uint32_t)(2 * (size_t)batch * kp) + (uint32_t)warp * 2 * buf_bytes;
    const uint32_t cap = (buf_bytes - 128) / 2 - 1;
    const int64_t T = 32 * (int64_t)M.steps;

    const int64_t gw = (int64_t)blockIdx.x * nwarp + warp, nw = (int64_t)gridDim.x * nwarp;
    RansTile cur{};
    if (gw < M.n_tiles) {
        cur = rans_tile(M, gw, make_uint2(__ldg(M.tile_off + gw), __ldg(M.tile_off + gw + 1)));
        rans_prefetch(bufs, cur, lane);
    }
    {
        const uint4* src = (const uint4*)M.table;
        uint4* dst = (uint4*)smem;
        for (int i = threadIdx.x; i < (int)(tab_bytes / 16); i += blockDim.x) dst[i] = __ldg(src + i);
    }
    grid_dep_launch();
    grid_dep_wait(); /* x, y and out belong to the preceding kernel in the stream from here on */
    if (kGemv) stage_x_rows(xs, a.x, batch, K, kp);
    __syncthreads();
    if (gw >= M.n_tiles) return;

    uint2 off_next = gw + nw < M.n_tiles ? make_uint2(__ldg(M.tile_off + gw + nw), __ldg(M.tile_off + gw + nw + 1))
                                         : make_uint2(0u, 0u);
    const uint32_t lt = (1u << lane) - 1u;
    uint32_t cb = bufs;
    for (int64_t t = gw; t < M.n_tiles; t += nw) {
        cp_async_wait_all();
        __syncwarp();
        const uint32_t nb_buf = cb == bufs ? bufs + buf_bytes : bufs;
        RansTile nxt{};
        if (t + nw < M.n_tiles) {
            nxt = rans_tile(M, t + nw, off_next);
            rans_prefetch(nb_buf, nxt, lane);
            if (t + 2 * nw < M.n_tiles)
                off_next = make_uint2(__ldg(M.tile_off + t + 2 * nw), __ldg(M.tile_off + t + 2 * nw + 1));
        }
        if (cur.words < 0) {
            if (lane == 0) flag_corrupt(a.status);
        } else {
            uint32_t x = lds32(cb + 4 * lane);
            const uint32_t wbase = cb + 128;
            uint32_t wp = 0;
            int64_t row = tile_row(t, T, kp, EC_RANS_ROW_ALIGN);
            uint32_t col = (uint32_t)(t * T - row * (int64_t)kp) + lane; /* this lane's column */
            float scale = __ldg(M.row_scales + row);
            float acc[B];
#pragma unroll
            for (int b = 0; b < B; ++b) acc[b] = 0.f;
            const uint32_t n_t = 32u * (uint32_t)cur.S;
            const uint32_t e_begin = __ldg(M.esc_off + t), e_end = __ldg(M.esc_off + t + 1);
            uint32_t er = e_begin; /* the tile's next record not yet folded in */
            /* the records of positions below p_end (the current row's end in the tile:
             * their weights were decoded as code 0, value 0, so each adds value * x),
             * then the warp's sums of the row, scaled by the row's r_i */
            auto flush = [&](uint32_t p_end) {
                const int64_t q0 = t * T - row * (int64_t)kp; /* column of tile position 0 in this row */
                while (er < e_end) {
                    const uint32_t j = er + (uint32_t)lane;
                    const uint32_t rec = j < e_end ? __ldg(M.esc + j) : 0xFFFFFFFFu, p = rec & 0xFFFFu;
                    const bool in = j < e_end && p < p_end;
                    if (in) {
                        if (p >= n_t) {
                            flag_corrupt(a.status);
                        } else {
                            const uint32_t c = (uint32_t)(q0 + p);
                            const float w = vals[256 + ((rec >> 16) & 0xFFu)];
#pragma unroll
                            for (int b = 0; b < B; ++b) {
                                if (B > 1 && b >= batch) break;
                                acc[b] = fmaf(w, __uint_as_float((uint32_t)xs[(size_t)b * kp + c] << 16), acc[b]);
                            }
                        }
                    }
                    const uint32_t nin = (uint32_t)__popc(__ballot_sync(kFull, in));
                    er += nin;
                    if (nin < 32) break;
                }
#pragma unroll
                for (int b = 0; b < B; ++b) {
                    if (B > 1 && b >= batch) break;
                    const float v = warp_sum(acc[b]) * scale;
                    if (lane == 0) {
                        float* dst = M.y + (int64_t)b * M.n_rows + row;
                        if (M.atomic_y) atomicAdd(dst, v);
                        else *dst = v;
                    }
                    acc[b] = 0.f;
                }
            };
            const int ng = cur.S / 4;
            for (int gi = 0; gi < ng; ++gi) {
                if (col >= kp) { /* rows start on 128-column boundaries */
                    if (kGemv) flush(128u * (uint32_t)gi);
                    col -= kp;
                    ++row;
                    scale = __ldg(M.row_scales + row);
                }
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                    const uint32_t e = lds32(tab_s + ((x & mask_b) << 2));
                    const uint32_t X = x >> pb;
                    x = (e >> 20) * X + X + ((e >> 8) & 0xFFFu); /* f X + bias with f - 1 in bits 20..31 */
                    const bool need = x < 65536u;
                    const uint32_t bal = __ballot_sync(kFull, need);
                    const uint32_t idx = min(wp + __popc(bal & lt), cap);
                    const uint32_t v = lds16_if(need, wbase + 2 * idx, 0u);
                    x = need ? x * 65536u + v : x;
                    wp += __popc(bal);
                    const float w = vals[e & 0xFFu];
                    const uint32_t c = col + 32 * s;
                    if (kGemv) {
#pragma unroll
                        for (int b = 0; b < B; ++b) {
                            if (B > 1 && b >= batch) break;
                            acc[b] = fmaf(w, __uint_as_float((uint32_t)xs[(size_t)b * kp + c] << 16), acc[b]);
                        }
                    } else if (c < K) {
                        M.out[row * K + c] = __bfloat16_as_ushort(__float2bfloat16_rn(__fmul_rn(w, scale)));
                    }
                }
                col += 128;
            }
            if (__any_sync(kFull, x != 65536u) || wp > (uint32_t)cur.words || (uint32_t)cur.words - wp > 7) {
                if (lane == 0) flag_corrupt(a.status);
            }
            if (kGemv) {
                flush(n_t);
            } else { /* the tile's corrections, after its own stores */
                __syncwarp();
                for (uint32_t e = e_begin + lane; e < e_end; e += 32) {
                    const uint32_t rec = __ldg(M.esc + e), p = rec & 0xFFFFu;
                    if (p >= n_t) {
                        flag_corrupt(a.status);
                        continue;
                    }
                    const int64_t q = t * T + p, r = q / (int64_t)kp, cc = q - r * (int64_t)kp;
                    if (cc >= K) continue;
                    const float w = vals[256 + ((rec >> 16) & 0xFFu)], sr = __ldg(M.row_scales + r);
                    M.out[r * K + cc] = __bfloat16_as_ushort(__float2bfloat16_rn(__fmul_rn(w, sr)));
                }
            }
        }
        cur = nxt;
        cb = nb_buf;
    }
}

/* ================================================== BF16 exponents through rANS */
/*
 * Kind 5 (MINE section 4, BF16 handling): the exponents of a tile's 32 lanes are
 * rANS symbols under a top-t table -- one exponent per symbol, or the exponents of
 * a lane's steps 2m and 2m + 1 ("Pair") -- and sign and mantissa are a plain byte
 * per weight, lane-transposed and pair-shuffled as in the Huffman tiles, so that
 * for every group of four lane steps one 32-bit word r holds [w(i+1) | w(i)] under
 * the mask 0x807F807F and [w(i+3) | w(i+2)] under the same mask after rotating by 8
 * bits.  A step: slot entry e = table[x mod 2^b], state update x = f (x >> b) +
 * (slot - cum), ballot + popc refill from the staged words (as the other rANS
 * kernels).  Single symbols carry the exponent in e's low byte; pair symbols index
 * a 256-entry table of exponent pairs already in BF16 position.
 *
 * GEMV: x sits in shared memory permuted per 128-column block, x'[128 k + 4 l + s] =
 * x[128 k + 32 s + l], so that lane l reads the x of its four steps in a block as
 * one 8-byte load; two FMA chains per batch row take the weight pairs.  A weight
 * whose exponent is outside the table was decoded with exponent 0; its record
 * (position | true BF16 << 16) adds (w - w_coded) x to the lane's sums before the
 * row's warp reduction, so no record needs an atomic of its own.
 */
template <bool kGemv, int B, bool kPair>
__global__ void __launch_bounds__(rans_max_warps(B) * 32, 1) exp_kernel(const __grid_constant__ ExpArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    const ExpMat& M = a.m;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarp = blockDim.x >> 5;
    const uint32_t kp = (uint32_t)M.k_pad;
    const int64_t K = M.k_cols;
    const int pb = M.prob_bits;
    const uint32_t mask_b = (1u << pb) - 1;
    const int batch = kGemv ? a.batch : 0;
    const uint32_t tab_s = smem_u32(smem), vals_s = tab_s + (4u << pb);
    const size_t tab_bytes = ((size_t)4 << pb) + 1024;
    uint16_t* xs = (uint16_t*)(smem + tab_bytes);
    const uint32_t xs_s = smem_u32(xs);
    const uint32_t buf_bytes = (uint32_t)rans_buf_bytes(M.words_cap);
    const uint32_t bufs = xs_s + (uint32_t)(2 * (size_t)batch * kp) + (uint32_t)warp * 2 * buf_bytes;
    const uint32_t cap = (buf_bytes - 128) / 2 - 1;
    const int64_t T = 32 * (int64_t)M.steps;

    const int64_t gw = (int64_t)blockIdx.x * nwarp + warp, nw = (int64_t)gridDim.x * nwarp;
    RansTile cur{};
    if (gw < M.n_tiles) {
        cur = rans_tile(M, gw, make_uint2(__ldg(M.tile_off + gw), __ldg(M.tile_off + gw + 1)));
        rans_prefetch(bufs, cur, lane);
    }
    {
        const uint4* src = (const uint4*)M.table;
        uint4* dst = (uint4*)smem;
        for (int i = threadIdx.x; i < (int)(tab_bytes / 16); i += blockDim.x) dst[i] = __ldg(src + i);
    }
    grid_dep_launch();
    grid_dep_wait(); /* x, y and out belong to the preceding kernel in the stream from here on */
    if (kGemv) stage_x_perm(xs, a.x, batch, K, kp);
    __syncthreads();
    if (gw >= M.n_tiles) return;

    uint2 off_next = gw + nw < M.n_tiles ? make_uint2(__ldg(M.tile_off + gw + nw), __ldg(M.tile_off + gw + nw + 1))
                                         : make_uint2(0u, 0u);
    const uint32_t lt = (1u << lane) - 1u;
    uint32_t cb = bufs;
    for (int64_t t = gw; t < M.n_tiles; t += nw) {
        cp_async_wait_all();
        __syncwarp();
        const uint32_t nb_buf = cb == bufs ? bufs + buf_bytes : bufs;
        RansTile nxt{};
        if (t + nw < M.n_tiles) {
            nxt = rans_tile(M, t + nw, off_next);
            rans_prefetch(nb_buf, nxt, lane);
            if (t + 2 * nw < M.n_tiles)
                off_next = make_uint2(__ldg(M.tile_off + t + 2 * nw), __ldg(M.tile_off + t + 2 * nw + 1));
        }
        if (cur.words < 0) {
            if (lane == 0) flag_corrupt(a.status);
        } else {
            uint32_t x = lds32(cb + 4 * lane);
            const uint32_t wbase = cb + 128;
            uint32_t wp = 0;
            int64_t row = tile_row(t, T, kp, EC_RANS_ROW_ALIGN);
            uint32_t col0 = (uint32_t)(t * T - row * (int64_t)kp); /* first column of the current 128-block */
            const uint32_t n_t = 32u * (uint32_t)cur.S;
            const uint32_t e_begin = __ldg(M.esc_off + t), e_end = __ldg(M.esc_off + t + 1);
            uint32_t er = e_begin; /* the tile's next record not yet folded in */
            float acc[B][2];
#pragma unroll
            for (int b = 0; b < B; ++b) acc[b][0] = acc[b][1] = 0.f;
            /* the records of positions below p_end (the current row's end in the tile),
             * then the warp's sums of the row */
            auto flush = [&](uint32_t p_end) {
                const int64_t q0 = t * T - row * (int64_t)kp; /* column of tile position 0 in this row */
                while (er < e_end) {
                    const uint32_t j = er + (uint32_t)lane;
                    const uint32_t rec = j < e_end ? __ldg(M.esc + j) : 0xFFFFFFFFu, p = rec & 0xFFFFu;
                    const bool in = j < e_end && p < p_end;
                    if (in) {
                        if (p >= n_t) {
                            flag_corrupt(a.status);
                        } else {
                            const uint32_t c = (uint32_t)(q0 + p), wt = rec >> 16, wd = wt & 0x807Fu;
#pragma unroll
                            for (int b = 0; b < B; ++b) {
                                if (B > 1 && b >= batch) break;
                                const uint32_t xv = xs[(size_t)b * kp + x_perm_index(c)];
                                acc[b][0] = fma1_bf16(wt, xv, acc[b][0]);
                                acc[b][1] = fma1_bf16(wd ^ 0x8000u, xv, acc[b][1]); /* - w_coded x */
                            }
                        }
                    }
                    const uint32_t nin = (uint32_t)__popc(__ballot_sync(kFull, in));
                    er += nin;
                    if (nin < 32) break;
                }
#pragma unroll
                for (int b = 0; b < B; ++b) {
                    if (B > 1 && b >= batch) break;
                    const float v = warp_sum(acc[b][0] + acc[b][1]);
                    if (lane == 0) {
                        float* dst = M.y + (int64_t)b * M.n_rows + row;
                        if (M.atomic_y) atomicAdd(dst, v);
                        else *dst = v;
                    }
                    acc[b][0] = acc[b][1] = 0.f;
                }
            };
            /* one rANS step: the slot entry of the decoded symbol */
            auto step = [&]() {
                const uint32_t e = lds32(tab_s + ((x & mask_b) << 2));
                const uint32_t X = x >> pb;
                x = (e >> 20) * X + X + ((e >> 8) & 0xFFFu);
                const bool need = x < 65536u;
                const uint32_t bal = __ballot_sync(kFull, need);
                const uint32_t idx = min(wp + __popc(bal & lt), cap);
                const uint32_t v = lds16_if(need, wbase + 2 * idx, 0u);
                x = need ? x * 65536u + v : x;
                wp += __popc(bal);
                return e;
            };
            const uint4* rawp = (const uint4*)(M.raw + t * (int64_t)M.raw_tile) + lane;
            const int ng = cur.S / 4; /* groups of four lane steps: 128 columns each */
            uint4 rq = __ldg(rawp), rn = ng > 4 ? __ldg(rawp + 32) : make_uint4(0u, 0u, 0u, 0u);
            for (int gi = 0; gi < ng; ++gi) {
                if (col0 >= kp) { /* rows start on 128-column boundaries */
                    if (kGemv) flush(128u * (uint32_t)gi);
                    col0 -= kp;
                    ++row;
                }
                const uint32_t r = (gi & 3) == 0 ? rq.x : (gi & 3) == 1 ? rq.y : (gi & 3) == 2 ? rq.z : rq.w;
                if ((gi & 3) == 3) {
                    rq = rn;
                    if (gi + 5 < ng) rn = __ldg(rawp + 32 * ((gi + 5) >> 2));
                }
                uint32_t E01, E23;
                if (kPair) {
                    E01 = lds32(vals_s + ((step() & 0xFFu) << 2));
                    E23 = lds32(vals_s + ((step() & 0xFFu) << 2));
                } else {
                    const uint32_t e0 = step() & 0xFFu, e1 = step() & 0xFFu, e2 = step() & 0xFFu, e3 = step() & 0xFFu;
                    E01 = (e0 << 7) | (e1 << 23);
                    E23 = (e2 << 7) | (e3 << 23);
                }
                const uint32_t W01 = (r & kSignMant) | E01, W23 = (__funnelshift_r(r, r, 8) & kSignMant) | E23;
                if (kGemv) {
#pragma unroll
                    for (int b = 0; b < B; ++b) {
                        if (B > 1 && b >= batch) break;
                        uint2 xv;
                        asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];"
                                     : "=r"(xv.x), "=r"(xv.y)
                                     : "r"(xs_s + 2u * ((uint32_t)b * kp + col0 + 4u * (uint32_t)lane)));
                        fma2x_bf16(W01, xv.x, acc[b][0], acc[b][1]);
                        fma2x_bf16(W23, xv.y, acc[b][0], acc[b][1]);
                    }
                } else {
                    const uint32_t c = col0 + (uint32_t)lane;
                    uint16_t* o = M.out + row * K;
                    if (c < K) o[c] = (uint16_t)W01;
                    if (c + 32 < K) o[c + 32] = (uint16_t)(W01 >> 16);
                    if (c + 64 < K) o[c + 64] = (uint16_t)W23;
                    if (c + 96 < K) o[c + 96] = (uint16_t)(W23 >> 16);
                }
                col0 += 128;
            }
            if (__any_sync(kFull, x != 65536u) || wp > (uint32_t)cur.words || (uint32_t)cur.words - wp > 7) {
                if (lane == 0) flag_corrupt(a.status);
            }
            if (kGemv) {
                flush(n_t);
            } else { /* the tile's records, after its own stores */
                __syncwarp();
                for (uint32_t e = e_begin + lane; e < e_end; e += 32) {
                    const uint32_t rec = __ldg(M.esc + e), p = rec & 0xFFFFu;
                    if (p >= n_t) {
                        flag_corrupt(a.status);
                        continue;
                    }
                    const int64_t q = t * T + p, rr = q / (int64_t)kp, cc = q - rr * (int64_t)kp;
                    if (cc < K) M.out[rr * K + cc] = (uint16_t)(rec >> 16);
                }
            }
        }
        cur = nxt;
        cb = nb_buf;
    }
}

/* ---- not in the Huffman GEMV: end ---- */
/* ======================================================== BF16 GEMV comparator */
constexpr int kRowsPerWarp = 4;

/* ---- E8 decode: begin ---- */
/* ======================================================= E8 lattice decode kernel */
/* EntroPack section 3.7: recover the coset and coordinate fields of every 8-weight
 * vector from independent rANS tiles, apply the algebraic inverse (z_8 from m and
 * the parity of z_1..z_7, q = 2 z + c), rescale by the shared and the row scale and
 * write BF16, with no intermediate symbol tensor and no reconstruction codebook.
 * One warp per tile; lane l owns the tile's vectors l, l + 32, ...: nine symbol
 * steps per vector (the coset first, then its 8 fields from the coset's tables),
 * each step a slot -> symbol lookup, the state update and a refill taken in lane
 * order (ballot + popc), as in the 4-bit kernel; the 8 weights of a vector are one
 * 16-byte store (a warp writes 512 contiguous bytes).
 *
 * Shared memory: the 17 slot -> symbol byte tables from a 2^PB-aligned address (so
 * a slot's address is one bitwise or), the 17 x 32 frequencies and the 17 x 32
 * starts as u16 arrays, then two tile buffers per warp. */
constexpr uint32_t kE8FreqBytes = 2u * EC_E8_TABLES * EC_E8_ALPHA; /* one u16 array: 1088 B */

__host__ __device__ constexpr size_t e8_table_bytes(int pb) {
    return ((size_t)1 << pb) /* alignment slack */ + ((size_t)EC_E8_TABLES << pb) + 2 * kE8FreqBytes;
}

__device__ __forceinline__ uint32_t e8_ld_sym(uint32_t addr) {
    uint32_t v;
    asm("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ uint2 e8_ld_freq(uint32_t addr) {
    uint2 v;
    asm("ld.shared.s16 %0, [%2];\n\tld.shared.u16 %1, [%2+%3];" : "=r"(v.x), "=r"(v.y) : "r"(addr), "n"(kE8FreqBytes));
    return v;
}

/* Bytes after the last tile buffer that a corrupt tile's refill reads may reach:
 * the read position is checked once per vector (9 steps of at most 32 words). */
constexpr uint32_t kE8Guard = 9 * 64;

/* Eight reconstructed values v_i = fp32(q_i g) / 2 in the output dtype: 0 = BF16,
 * 1 = FP8 E4M3 (nearest, ties to even, saturating), 2 = INT8 (same rounding). */
template <int OUT>
__device__ __forceinline__ void e8_store(void* out, int64_t at, const float (&v)[8]) {
    if constexpr (OUT == 0) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
            w[i] = *(const uint32_t*)&h;
        }
        *(uint4*)((uint16_t*)out + at) = make_uint4(w[0], w[1], w[2], w[3]);
    } else if constexpr (OUT == 1) {
        uint32_t h[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            h[i] = __nv_cvt_float2_to_fp8x2(make_float2(v[2 * i], v[2 * i + 1]), __NV_SATFINITE, __NV_E4M3);
        *(uint2*)((uint8_t*)out + at) = make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
    } else {
        uint32_t b[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) b[i] = (uint32_t)min(127, max(-128, __float2int_rn(v[i]))) & 0xFFu;
        *(uint2*)((uint8_t*)out + at) =
            make_uint2(b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24), b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24));
    }
}

template <int PB, int OUT>
__global__ void __launch_bounds__(kMaxHW * 32, 1) e8_kernel(const __grid_constant__ E8Args a) {
    extern __shared__ __align__(16) uint8_t smem[];
    const E8Mat& M = a.m;
    constexpr uint32_t kSlots = 1u << PB, kMask = kSlots - 1;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarp = blockDim.x >> 5;
    const uint32_t base = smem_u32(smem);
    const uint32_t pad = (kSlots - (base & kMask)) & kMask; /* a multiple of 16 */
    uint8_t* const ss = smem + pad;
    const uint32_t ss_s = base + pad, fq_s = ss_s + EC_E8_TABLES * kSlots;
    const uint32_t buf_bytes = (uint32_t)rans_buf_bytes(M.words_cap);
    const uint32_t bufs = base + (uint32_t)e8_table_bytes(PB) + (uint32_t)(warp * a.nbuf) * buf_bytes;
    const bool dbl = a.nbuf == 2;
    const int64_t T = 32 * (int64_t)M.steps; /* vectors per tile */
    const int64_t vpr = M.k_pad / 8, K = M.k_cols;

    const int64_t gw = (int64_t)blockIdx.x * nwarp + warp, nw = (int64_t)gridDim.x * nwarp;
    RansTile cur{};
    if (gw < M.n_tiles) {
        cur = rans_tile(M, gw, make_uint2(__ldg(M.tile_off + gw), __ldg(M.tile_off + gw + 1)));
        rans_prefetch(bufs, cur, lane);
    }
    {
        const uint4* s2 = (const uint4*)M.slot_sym;
        uint4* d2 = (uint4*)ss;
        for (uint32_t i = threadIdx.x; i < EC_E8_TABLES * kSlots / 16; i += blockDim.x) d2[i] = __ldg(s2 + i);
        /* per table and symbol: f - 2^PB (so that x' = x + (x >> PB)(f - 2^PB) - start) and the start */
        int16_t* fq = (int16_t*)(ss + EC_E8_TABLES * kSlots);
        for (uint32_t i = threadIdx.x; i < EC_E8_TABLES * EC_E8_ALPHA; i += blockDim.x) {
            const uint32_t e = __ldg(M.fc + i);
            fq[i] = (int16_t)((int32_t)(e & 0xFFFFu) - (int32_t)kSlots);
            fq[EC_E8_TABLES * EC_E8_ALPHA + i] = (int16_t)(e >> 16);
        }
    }
    grid_dep_launch();
    grid_dep_wait(); /* out belongs to the preceding kernel in the stream from here on */
    __syncthreads();
    if (gw >= M.n_tiles) return;

    uint2 off_next = gw + nw < M.n_tiles ? make_uint2(__ldg(M.tile_off + gw + nw), __ldg(M.tile_off + gw + nw + 1))
                                         : make_uint2(0u, 0u);
    const uint32_t lt = (1u << lane) - 1u;
    const uint32_t f0 = __ldg(M.fc) & 0xFFFFu, nf0 = f0 - kSlots, nf1 = (__ldg(M.fc + 1) & 0xFFFFu) - kSlots;
    uint32_t cb = bufs;
    for (int64_t t = gw; t < M.n_tiles; t += nw) {
        cp_async_wait_all();
        __syncwarp();
        /* two buffers: the next tile streams into the other one during this decode;
         * one buffer: it is loaded after this decode (other warps hide the wait) */
        const uint32_t nb_buf = dbl ? (cb == bufs ? bufs + buf_bytes : bufs) : bufs;
        RansTile nxt{};
        if (t + nw < M.n_tiles) {
            nxt = rans_tile(M, t + nw, off_next);
            if (dbl) rans_prefetch(nb_buf, nxt, lane);
            if (t + 2 * nw < M.n_tiles)
                off_next = make_uint2(__ldg(M.tile_off + t + 2 * nw), __ldg(M.tile_off + t + 2 * nw + 1));
        }
        if (cur.words < 0) {
            if (lane == 0) flag_corrupt(a.status);
        } else {
            uint32_t x = ((const uint32_t*)(smem + (cb - base)))[lane];
            const uint32_t w0 = cb + 128, wlim = w0 + 2 * (uint32_t)M.words_cap;
            uint32_t wa = w0; /* shared address of the next unread payload word */
            const int64_t v0 = t * T + lane;
            int64_t row = v0 / vpr;
            int64_t cv = v0 - row * vpr; /* this lane's vector column */
            float g = __fmul_rn(M.scale, __ldg(M.row_scales + row));
            bool bad = false;
            /* the refill after a symbol: lanes whose state fell below 2^16 take the next
             * words in lane order */
            auto refill = [&]() {
                const bool need = x < 65536u;
                const uint32_t bal = __ballot_sync(kFull, need);
                const uint32_t v = lds16(wa + 2 * __popc(bal & lt));
                x = need ? (x << 16) | v : x;
                wa += 2 * __popc(bal);
            };
            /* one symbol: tab = the table's 2^PB-aligned slot base, fq = its frequency row */
            auto step = [&](uint32_t tab, uint32_t fq) {
                const uint32_t sym = e8_ld_sym(tab | (x & kMask));
                const uint2 fc = e8_ld_freq(fq + 2 * sym); /* (f - 2^PB) sign-extended, start */
                x = (x >> PB) * fc.x + (x - fc.y);
                refill();
                return sym;
            };
            for (int j = 0; j < cur.S; ++j) {
                if (wa > wlim) { /* warp-uniform: only a corrupt tile reads past its words */
                    bad = true;
                    break;
                }
                /* the coset: table 0 holds symbols 0 and 1 only, so the slot's side of
                 * start(1) = f(0) decides it, with no table lookup */
                const uint32_t c = (x & kMask) >= f0 ? 1u : 0u;
                x = (x >> PB) * (c ? nf1 : nf0) + (x - (c ? f0 : 0u));
                refill();
                const uint32_t tab = ss_s + ((1u + 8u * c) << PB), fq = fq_s + (1u + 8u * c) * 2u * EC_E8_ALPHA;
                uint32_t s[8];
#pragma unroll
                for (int f = 0; f < 8; ++f) s[f] = step(tab + ((uint32_t)f << PB), fq + 2u * EC_E8_ALPHA * f);
                /* z_j = s_j - 16; z_8 = 2 m + parity(z_1..z_7) with m = s_8 - 16; q = 2 z + c */
                const uint32_t par = (s[0] ^ s[1] ^ s[2] ^ s[3] ^ s[4] ^ s[5] ^ s[6]) & 1u;
                int q[8];
#pragma unroll
                for (int f = 0; f < 7; ++f) q[f] = 2 * (int)s[f] - 32 + (int)c;
                q[7] = 4 * (int)s[7] - 64 + 2 * (int)par + (int)c;
                float v[8];
                /* fl(fl(q g) / 2) == fl(q (g / 2)) while g / 2 is normal and q g finite
                 * (|q| <= 32): one rounding either way; otherwise both multiplies */
                const float ag = fabsf(g);
                if (ag >= 0x1p-125f && ag <= 0x1p120f) {
                    const float gh = g * 0.5f;
#pragma unroll
                    for (int i = 0; i < 8; ++i) v[i] = __fmul_rn(__int2float_rn(q[i]), gh);
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) v[i] = __fmul_rn(__fmul_rn(__int2float_rn(q[i]), g), 0.5f);
                }
                if (8 * cv < K) e8_store<OUT>(M.out, row * K + 8 * cv, v);
                cv += 32;
                if (cv >= vpr) {
                    cv -= vpr;
                    ++row;
                    if (j + 1 < cur.S) g = __fmul_rn(M.scale, __ldg(M.row_scales + row));
                }
            }
            /* every lane returns to 2^16 and the words are used up (up to 7 padding words) */
            const uint32_t used = (wa - w0) / 2;
            if (bad || __any_sync(kFull, x != 65536u) || used > (uint32_t)cur.words || (uint32_t)cur.words - used > 7) {
                if (lane == 0) flag_corrupt(a.status);
            }
        }
        if (!dbl && t + nw < M.n_tiles) {
            __syncwarp(); /* every lane has read the buffer before it is overwritten */
            rans_prefetch(bufs, nxt, lane);
        }
        cur = nxt;
        cb = nb_buf;
    }
}

/* ---- E8 decode: end ---- */

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

/* Smallest batch that the Huffman GEMV runs on the tensor cores (when the
 * matrices' tiles lie inside rows); EC_MMA_MIN_BATCH overrides it (a value above
 * EC_MAX_BATCH keeps every batch on the CUDA cores). */
int mma_min_batch() {
    static const int v = [] {
        const char* e = std::getenv("EC_MMA_MIN_BATCH");
        return e && e[0] ? std::max(1, std::atoi(e)) : 6;
    }();
    return v;
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
    m.n_sub = h.huff_sub_tables;
    m.sub_smem = -1;
    m.fill = h.huff_fill;
    m.n_rows = h.n_rows;
    m.k_cols = h.k_cols;
    m.k_pad = h.k_pad;
    m.out_ld = h.k_cols;
    m.n_tiles = h.n_tiles;
    m.records_bytes = h.blob_bytes - h.records_off;
    m.steps = h.steps;
    const int64_t T = 32 * (int64_t)h.steps;
    m.atomic_y = (h.k_pad > 0 && T % h.k_pad == 0) ? 0 : 1;
    m.last_steps = h.n_tiles > 0 ? (int32_t)((h.n_rows * h.k_pad - (h.n_tiles - 1) * T) / 32) : 0;
    m.rec16 = (uint32_t)(m.records_bytes / 16);
    return m;
}

/* ---- not in the Huffman GEMV: begin ---- */
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
    m.last_steps = h.n_tiles > 0 ? (int32_t)((h.n_rows * h.k_pad - (h.n_tiles - 1) * T) / 32) : 0;
    m.rec16 = (uint32_t)(m.records_bytes / 16);
    m.tuple = h.rans_tuple;
    m.values = h.rans_values;
    return m;
}
/* ---- not in the Huffman GEMV: end ---- */

Fp8Mat fp8_desc(const ec_matrix* W) {
    Fp8Mat m{};
    const ec_blob_header& h = W->hdr;
    m.records = W->d_blob + h.records_off;
    m.tile_off = (const uint32_t*)(W->d_blob + h.tile_off_off);
    m.table = (const uint32_t*)(W->d_blob + h.table_off);
    m.row_scales = (const float*)(W->d_blob + h.scales_off);
    m.esc_off = (const uint32_t*)(W->d_blob + h.esc_off_off);
    m.esc = (const uint32_t*)(W->d_blob + h.esc_records_off);
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
    m.last_steps = h.n_tiles > 0 ? (int32_t)((h.n_rows * h.k_pad - (h.n_tiles - 1) * T) / 32) : 0;
    m.rec16 = (uint32_t)(m.records_bytes / 16);
    return m;
}

ExpMat exp_desc(const ec_matrix* W) {
    ExpMat m{};
    const ec_blob_header& h = W->hdr;
    m.records = W->d_blob + h.records_off;
    m.tile_off = (const uint32_t*)(W->d_blob + h.tile_off_off);
    m.table = (const uint32_t*)(W->d_blob + h.table_off);
    m.raw = W->d_blob + h.scales_off;
    m.esc_off = (const uint32_t*)(W->d_blob + h.esc_off_off);
    m.esc = (const uint32_t*)(W->d_blob + h.esc_records_off);
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
    m.last_steps = h.n_tiles > 0 ? (int32_t)((h.n_rows * h.k_pad - (h.n_tiles - 1) * T) / 32) : 0;
    m.rec16 = (uint32_t)(m.records_bytes / 16);
    m.raw_tile = EC_RAW_BYTES(h.steps);
    m.tuple = h.rans_tuple;
    return m;
}

/* ---- E8 decode: begin ---- */
E8Mat e8_desc(const ec_matrix* W) {
    E8Mat m{};
    const ec_blob_header& h = W->hdr;
    m.records = W->d_blob + h.records_off;
    m.tile_off = (const uint32_t*)(W->d_blob + h.tile_off_off);
    m.fc = (const uint32_t*)(W->d_blob + h.table_off);
    m.slot_sym = W->d_blob + h.table_off + 4 * EC_E8_TABLES * EC_E8_ALPHA;
    m.row_scales = (const float*)(W->d_blob + h.scales_off);
    m.n_rows = h.n_rows;
    m.k_cols = h.k_cols;
    m.k_pad = h.k_pad;
    m.n_tiles = h.n_tiles;
    m.records_bytes = h.blob_bytes - h.records_off;
    m.steps = h.steps;
    m.prob_bits = h.prob_bits;
    m.words_cap = (h.max_words + 7) / 8 * 8;
    const int64_t T = 32 * (int64_t)h.steps, n_vec = h.n_rows * (h.k_pad / 8);
    m.last_steps = h.n_tiles > 0 ? (int32_t)((n_vec - (h.n_tiles - 1) * T) / 32) : 0;
    m.rec16 = (uint32_t)(m.records_bytes / 16);
    std::memcpy(&m.scale, &h.e8_scale_bits, 4);
    return m;
}
/* ---- E8 decode: end ---- */

int check_matrix(const ec_matrix* W, int dev) {
    if (!W || !W->d_blob || W->hdr.magic != EC_BLOB_MAGIC || W->hdr.version != EC_BLOB_VERSION) return EC_ERR_INVALID_ARG;
    if (W->device != dev) return EC_ERR_INVALID_ARG;
    /* the Huffman kernels keep tile, row and column indices in 32 bits: a launch of
     * up to EC_MAX_GROUP (or EC_MAX_DECODE_BATCH) such matrices stays below 2^31 tiles */
    if (W->kind == EC_KIND_HUFFMAN_BF16 &&
        (W->hdr.n_tiles > (int64_t(1) << 24) || W->hdr.n_rows >= (int64_t(1) << 31) || W->hdr.k_pad >= (int64_t(1) << 31)))
        return EC_ERR_UNSUPPORTED;
    return EC_OK;
}

/* Largest number of warps' worth of per-warp buffers that fits next to `fixed`. */
int grid_for(const DeviceInfo& d, int64_t work_items, int ctas_per_sm) {
    const int64_t full = (int64_t)d.sms * ctas_per_sm;
    const int64_t need = (work_items + kWarps - 1) / kWarps;
    return (int)std::max<int64_t>(1, std::min(full, need));
}

/* Room of a per-warp tile buffer for matrix W (after the 64 bytes of lane starts):
 * its largest code area and kStagedRecs window records; a tile's further records
 * are read from global memory. */
constexpr int kStagedRecs = 64;
int staged_code_bytes(const ec_matrix* W) {
    const int area = (W->hdr.max_code_area + 15) & ~15;
    return std::min(area + 4 * kStagedRecs, std::max(area, (W->hdr.max_code_bytes + 15) & ~15));
}

/* A matrix decoded through the hierarchical tables (no window records). */
bool huff_hier(const ec_matrix* W) { return !(W->hdr.huff_flags & EC_HUFF_WINDOW_REC); }

/* Stage the sub-tables of a launch's hierarchical matrices in shared memory, in
 * order, while kSubSmemTables hold them; returns the staged words. */
template <int N>
int plan_sub_tables(HuffMat (&m)[N], int count) {
    int used = 0;
    for (int k = 0; k < count; ++k) {
        m[k].sub_smem = -1;
        if (m[k].n_sub == 0) continue;
        if (used + m[k].n_sub <= kSubSmemTables) {
            m[k].sub_smem = 256 * used;
            used += m[k].n_sub;
        }
    }
    return 256 * used;
}

/* kPart selects the allocation-free variant, lng (hierarchical) the kernel that
 * checks every pair and walks the sub-tables for what the window cannot hold. */
template <int B, bool kPart>
int launch_huff_gemv_b(const HuffGemvArgs& a, bool lng, size_t smem, int grid, int block, cudaStream_t s) {
    auto kern = lng ? huff_gemv_kernel<B, kPart, true, false> : huff_gemv_kernel<B, kPart, false, false>;
    if (B == 1 && !kPart && a.tx_cols > 0)
        kern = lng ? huff_gemv_kernel<1, false, true, true> : huff_gemv_kernel<1, false, false, true>;
    if (set_smem(kern, smem) != EC_OK) return EC_ERR_CUDA;
    return launch_ex(kern, grid, block, smem, s, a);
}

template <bool kPart>
int launch_huff_gemv(const HuffGemvArgs& a, bool lng, size_t smem, int grid, int block, cudaStream_t s) {
    if (a.batch <= 1) return launch_huff_gemv_b<1, kPart>(a, lng, smem, grid, block, s);
    if (a.batch <= 2) return launch_huff_gemv_b<2, kPart>(a, lng, smem, grid, block, s);
    if (a.batch <= 4) return launch_huff_gemv_b<4, kPart>(a, lng, smem, grid, block, s);
    if (a.batch <= 8) return launch_huff_gemv_b<8, kPart>(a, lng, smem, grid, block, s);
    return launch_huff_gemv_b<16, kPart>(a, lng, smem, grid, block, s);
}

/* ---- not in the Huffman GEMV: begin ---- */
template <bool G, int B>
int launch_rans_b(const RansArgs& a, size_t smem, int grid, int block, cudaStream_t s) {
    auto kern = a.m.tuple == 2 ? rans_kernel<G, B, true> : rans_kernel<G, B, false>;
    if (set_smem(kern, smem) != EC_OK) return EC_ERR_CUDA;
    return launch_ex(kern, grid, block, smem, s, a);
}

int launch_rans(bool gemv, const RansArgs& a, size_t smem, int grid, int block, cudaStream_t s) {
    if (!gemv) return launch_rans_b<false, 1>(a, smem, grid, block, s);
    if (a.batch <= 1) return launch_rans_b<true, 1>(a, smem, grid, block, s);
    if (a.batch <= 2) return launch_rans_b<true, 2>(a, smem, grid, block, s);
    if (a.batch <= 4) return launch_rans_b<true, 4>(a, smem, grid, block, s);
    if (a.batch <= 8) return launch_rans_b<true, 8>(a, smem, grid, block, s);
    return launch_rans_b<true, 16>(a, smem, grid, block, s);
}
/* ---- not in the Huffman GEMV: end ---- */

/* Batch rows whose copy of x (elem bytes per value) fits in `budget` bytes of shared memory. */
int rows_per_pass(int64_t k_pad, int batch, size_t budget, int elem = 4) {
    if (k_pad == 0) return batch;
    const int64_t per = elem * k_pad;
    return (int)std::max<int64_t>(0, std::min<int64_t>(batch, (int64_t)budget / per));
}

/* ----------------------------------------------------------- Huffman GEMV */
/* Launch shape of a Huffman GEMV: warps per CTA (as many as fit next to the pair
 * tables and one batch row of x, capped by the kernel's register budget for the
 * batch width), batch rows per pass, one CTA per SM at most. */
struct GemvPlan {
    int warps, per_pass, grid;
    size_t fixed, xrow;
};

/* Rows and columns between a tile and the one `warps_total` tiles later. */
void set_tile_stride(HuffMat& m, int64_t warps_total) {
    const int64_t span = warps_total * 32 * (int64_t)m.steps;
    m.d_row = m.k_pad > 0 ? span / m.k_pad : 0;
    m.d_col = m.k_pad > 0 ? span % m.k_pad : 0;
}

int plan_huff_gemv(const DeviceInfo& d, int count, int code_bytes, int64_t kp, int batch, int64_t total_tiles,
                   int sub_words, GemvPlan* pl) {
    /* the TMEM address slot (16 B), the pair tables and the staged sub-tables */
    const size_t tables = 16 + (size_t)count * kPairTabBytes + 4 * (size_t)sub_words, per_warp = huff_warp_bytes(code_bytes);
    pl->xrow = xs_row_bytes((uint32_t)kp);
    if (tables + pl->xrow + 4 * per_warp > d.smem_optin) return EC_ERR_UNSUPPORTED;
    const int cap = huff_max_warps(batch <= 1 ? 1 : batch <= 2 ? 2 : batch <= 4 ? 4 : batch <= 8 ? 8 : 16);
    const int wmax = (int)std::min<size_t>(cap, (d.smem_optin - tables - pl->xrow) / per_warp);
    /* Each warp takes every (grid * warps)-th tile, grid = min(SMs, tiles / w): an
     * SM runs tiles / grid tiles in rounds of w warps, the last round with what is
     * left.  A round takes time in proportion to its busy warps, but no less than
     * with 16 (below that the warps' decode chains leave the SM idle).  Batch rows
     * whose x does not fit next to the warps' buffers take further passes, each
     * decoding the matrices again.  Cost = passes * sum over rounds of max(busy,
     * 16); among the w within 1 % of the cheapest take the one with the largest
     * grid, then the largest w. */
    constexpr double kFloor = 16.0;
    double cost[33] = {};
    int rows_of[33] = {};
    int64_t grid_of[33] = {};
    double best_cost = 1e300;
    for (int w = 1; w <= wmax; ++w) {
        const size_t fixed = tables + (size_t)w * per_warp;
        const int rows = (int)std::min<size_t>(std::min(batch, kFmaMaxRows), (d.smem_optin - fixed) / pl->xrow);
        const int64_t passes = (batch + rows - 1) / rows;
        const int64_t g = std::max<int64_t>(1, std::min<int64_t>(d.sms, (total_tiles + w - 1) / w));
        const double per_sm = (double)total_tiles / (double)g; /* tiles (warp rounds) each SM runs */
        const int64_t rounds = (int64_t)std::ceil(per_sm / w - 1e-9);
        const double last = per_sm - (double)(rounds - 1) * w; /* warps busy in the last round */
        cost[w] = (double)passes * ((double)(rounds - 1) * std::max<double>(w, kFloor) + std::max(last, kFloor));
        rows_of[w] = rows;
        grid_of[w] = g;
        best_cost = std::min(best_cost, cost[w]);
    }
    int best = wmax, best_rows = rows_of[wmax];
    int64_t best_grid = -1;
    for (int w = wmax; w >= 1; --w)
        if (cost[w] <= 1.01 * best_cost && grid_of[w] > best_grid) {
            best = w;
            best_rows = rows_of[w];
            best_grid = grid_of[w];
        }
    pl->warps = best;
    pl->fixed = tables + (size_t)pl->warps * per_warp;
    pl->per_pass = best_rows;
    pl->grid = (int)std::max<int64_t>(1, std::min<int64_t>(d.sms, (total_tiles + pl->warps - 1) / pl->warps));
    return EC_OK;
}


/* Tensor-core path: every matrix's tiles must lie inside one row. */
bool mma_layout(const ec_matrix* W) {
    const ec_blob_header& h = W->hdr;
    return h.n_tiles > 0 && h.steps % 16 == 0 && h.k_pad % (32 * (int64_t)h.steps) == 0 && h.k_pad < (int64_t(1) << 31) &&
           h.window_code_bytes > 0;
}

/* cuTensorMapEncodeTiled, reached through the runtime (no link against the driver library). */
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return (PFN_cuTensorMapEncodeTiled_v12000)p;
    }();
    return fn;
}

/* x [rows, K] BF16 as TMA boxes of 32 rows x 64 columns (128 bytes) with the
 * 128-byte swizzle of the MMA operand; rows past `rows` and columns past K read
 * as zero.  Needs K % 8 == 0 (16-byte row stride) and a 16-byte aligned x. */
int encode_x_map(CUtensorMap* map, const uint16_t* x, int64_t K, int rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return EC_ERR_CUDA;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {64, 32}, estr[2] = {1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (void*)x, dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? EC_OK : EC_ERR_CUDA;
}

/* Whether the tensor-core kernel's fixed shared memory (two chunk buffers, the pair
 * tables, the staged sub-tables and two pools of one item's code areas) fits the
 * 227 KB a block may have on sm_103a (the same sums as huff_mma makes). */
bool mma_fits(const ec_matrix* const* Ws, int count) {
    int used = 0;
    int64_t window = 0;
    for (int k = 0; k < count; ++k) {
        const int n = Ws[k]->hdr.huff_sub_tables;
        if (n > 0 && used + n <= kSubSmemTables) used += n;
        window = std::max<int64_t>(window, Ws[k]->hdr.window_code_bytes);
    }
    const size_t fixed = mma_fixed_bytes(2) + (size_t)count * kPairTabBytes + 4 * 256 * (size_t)used +
                         2 * (size_t)((window + 15) & ~int64_t(15));
    return fixed <= 232448;
}

/* Huffman GEMVs from mma_min_batch() on, on matrices whose tiles lie inside rows and
 * rows of x that TMA can address (16-byte stride), take the tensor-core kernel when
 * its buffers fit (not for the widest tiles of long rows). */
bool use_mma(const ec_matrix* const* Ws, int count, int batch) {
    bool mma = batch >= mma_min_batch() && Ws[0]->hdr.k_cols % 8 == 0;
    for (int k = 0; k < count && mma; ++k) mma = mma_layout(Ws[k]);
    return mma && mma_fits(Ws, count);
}

/* ---- not in the Huffman GEMV: begin ---- */
int huff_mma(const ec_matrix* const* Ws, int count, const uint16_t* x, float* const* ys, int batch, cudaStream_t s,
             DeviceInfo* d) {
    HuffMmaArgs a{};
    a.count = count;
    a.status = d->status;
    int code_bytes = 16;
    bool lng = false;
    int64_t total = 0;
    const int64_t K = Ws[0]->hdr.k_cols;
    for (int k = 0; k < count; ++k) {
        const ec_matrix* W = Ws[k];
        a.m[k] = huff_desc(W);
        a.m[k].tile_begin = total;
        total += W->hdr.n_tiles;
        a.row_tiles[k] = (int32_t)(W->hdr.k_pad / (32 * (int64_t)W->hdr.steps));
        code_bytes = std::max(code_bytes, (int)W->hdr.max_code_bytes);
        lng = lng || huff_hier(W);
        if (a.m[k].atomic_y &&
            cudaMemsetAsync(ys[k], 0, sizeof(float) * (size_t)batch * (size_t)W->hdr.n_rows, s) != cudaSuccess)
            return EC_ERR_CUDA;
    }
    a.sub_words = plan_sub_tables(a.m, count);
    code_bytes = (code_bytes + 15) & ~15;
    a.code_bytes = code_bytes;
    a.total_tiles = total;
    /* one item's tiles, packed: the largest window of EC_MMA_WINDOW_ROWS rows, plus slack */
    int64_t window = 0;
    for (int k = 0; k < count; ++k) window = std::max<int64_t>(window, Ws[k]->hdr.window_code_bytes);
    a.pool_bytes = (int)((window + 15) & ~int64_t(15));
    /* warps: a multiple of 8, at most 32 (one produces, the others decode one row each:
     * rows per item = warps - 1 <= EC_MMA_WINDOW_ROWS, N = warps); 3 chunk buffers where they fit */
    const size_t fixed_rest = (size_t)count * kPairTabBytes + 4 * (size_t)a.sub_words + 2 * (size_t)a.pool_bytes;
    int nw = 0, nbuf = 0;
    for (int nb = kMmaMaxBufs; nb >= 2 && !nw; --nb)
        for (int w = kMaxHW; w >= (nb == 2 ? 8 : kMaxHW) && !nw; w -= 8)
            if (mma_fixed_bytes(nb) + fixed_rest <= d->smem_optin) {
                nw = w;
                nbuf = nb;
            }
    if (!nw) return EC_ERR_UNSUPPORTED;
    a.nbuf = nbuf;
    const int rows = nw - 1;
    const size_t smem = mma_fixed_bytes(nbuf) + fixed_rest;
    a.item_begin[0] = 0;
    for (int k = 0; k < count; ++k)
        a.item_begin[k + 1] = a.item_begin[k] + (Ws[k]->hdr.n_rows + rows - 1) / rows * a.row_tiles[k];
    /* kind::f16 instruction descriptor: FP32 accumulators (bits 4..5 = 1), BF16 A and B
     * (bits 7..9, 10..12 = 1), both K-major, N >> 3 in bits 17..22, M >> 4 in bits 24..28 */
    a.idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(nw >> 3) << 17) | ((64u >> 4) << 24);
    const int grid = (int)std::min<int64_t>(d->sms, a.item_begin[count]);
    auto kern = lng ? huff_mma_kernel<true> : huff_mma_kernel<false>;
    if (set_smem(kern, smem) != EC_OK) return EC_ERR_CUDA;
    for (int b0 = 0; b0 < batch; b0 += kMmaMaxBatch) {
        a.batch = std::min(kMmaMaxBatch, batch - b0);
        int rc = encode_x_map(&a.xmap, x + (int64_t)b0 * K, K, a.batch);
        if (rc != EC_OK) return rc;
        for (int k = 0; k < count; ++k) a.m[k].y = ys[k] + (int64_t)b0 * Ws[k]->hdr.n_rows;
        if ((rc = launch_ex(kern, grid, nw * 32, smem, s, a)) != EC_OK) return rc;
    }
    return EC_OK;
}
/* ---- not in the Huffman GEMV: end ---- */

int huff_gemv(const ec_matrix* const* Ws, int count, const uint16_t* x, float* const* ys, int batch,
              cudaStream_t s, int dev, DeviceInfo* d) {
    if (use_mma(Ws, count, batch)) return huff_mma(Ws, count, x, ys, batch, s, d);
    int64_t total = 0;
    int code_bytes = 16;
    bool lng = false;
    HuffGemvArgs a{};
    a.count = count;
    const int64_t K = Ws[0]->hdr.k_cols, kp = Ws[0]->hdr.k_pad;
    for (int k = 0; k < count; ++k) {
        const ec_matrix* W = Ws[k];
        a.m[k] = huff_desc(W);
        a.m[k].tile_begin = total;
        total += W->hdr.n_tiles;
        code_bytes = std::max(code_bytes, staged_code_bytes(W));
        lng = lng || huff_hier(W);
        if (a.m[k].atomic_y || W->hdr.n_tiles == 0) {
            if (cudaMemsetAsync(ys[k], 0, sizeof(float) * (size_t)batch * (size_t)W->hdr.n_rows, s) != cudaSuccess)
                return EC_ERR_CUDA;
        }
    }
    code_bytes = (code_bytes + 15) & ~15;
    a.total_tiles = total;
    a.status = d->status;
    a.code_bytes = code_bytes;
    a.sub_words = plan_sub_tables(a.m, count);
    if (total == 0) return EC_OK;
    GemvPlan pl;
    int rc = plan_huff_gemv(*d, count, code_bytes, kp, batch, total, a.sub_words, &pl);
    if (rc != EC_OK) return rc;
    for (int k = 0; k < count; ++k) set_tile_stride(a.m[k], (int64_t)pl.grid * pl.warps);
    /* batch 1 over tiles that lie inside rows, all of one width: x from tensor memory */
    if (batch == 1) {
        const int64_t T = 32 * (int64_t)Ws[0]->hdr.steps;
        bool ok = T > 0 && kp % T == 0;
        for (int k = 0; k < count && ok; ++k) ok = Ws[k]->hdr.steps == Ws[0]->hdr.steps;
        const int64_t used = ok ? (kp / T) * (T / 64) : 0;
        int cols = 32;
        while (cols < used + 8) cols *= 2; /* + 8: the load past a tile's last block */
        if (ok && used > 0 && cols <= 512) {
            a.tx_cols = cols;
            a.tx_layout_cols = (int)(T / 64);
            a.tx_used = (int)used;
            a.tx_T = (uint32_t)T;
        }
    }
    for (int b0 = 0; b0 < batch; b0 += pl.per_pass) {
        const int nb = std::min(pl.per_pass, batch - b0);
        a.batch = nb;
        a.x = x + (int64_t)b0 * K;
        for (int k = 0; k < count; ++k) a.m[k].y = ys[k] + (int64_t)b0 * Ws[k]->hdr.n_rows;
        if ((rc = launch_huff_gemv<false>(a, lng, pl.fixed + pl.xrow * nb, pl.grid, pl.warps * 32, s)) != EC_OK)
            return rc;
    }
    return EC_OK;
}

/* ---- not in the Huffman GEMV: begin ---- */
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
    /* one CTA per SM: slot table | (GEMV) code-pair table | x (BF16) [rows of this pass][k_pad] |
     * two tile buffers per warp */
    const size_t table = ((size_t)4 << a.m.prob_bits) + (gemv ? 1024 : 0), per_warp = 2 * rans_buf_bytes(a.m.words_cap);
    const int64_t kp = W->hdr.k_pad, K = W->hdr.k_cols;
    const size_t xrow = gemv ? (size_t)2 * kp : 0;
    if (table + xrow + 4 * per_warp > d->smem_optin) return EC_ERR_UNSUPPORTED;
    const int cap = gemv ? rans_max_warps(batch <= 1 ? 1 : batch <= 2 ? 2 : batch <= 4 ? 4 : batch <= 8 ? 8 : 16)
                         : rans_max_warps(1);
    const int warps = (int)std::min<size_t>(cap, (d->smem_optin - table - xrow) / per_warp);
    const size_t fixed = table + (size_t)warps * per_warp;
    const int per_pass = gemv ? (int)std::min<size_t>(std::min(batch, kFmaMaxRows), (d->smem_optin - fixed) / xrow) : 1;
    if (per_pass < 1) return EC_ERR_UNSUPPORTED;
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(d->sms, (W->hdr.n_tiles + warps - 1) / warps));
    const int passes = gemv ? batch : 1;
    for (int b0 = 0; b0 < passes; b0 += per_pass) {
        const int nb = gemv ? std::min(per_pass, batch - b0) : 0;
        a.batch = nb;
        a.x = gemv ? x + (int64_t)b0 * K : nullptr;
        if (gemv) a.m.y = y + (int64_t)b0 * W->hdr.n_rows;
        const int rc = launch_rans(gemv, a, fixed + xrow * nb, grid, warps * 32, s);
        if (rc != EC_OK) return rc;
    }
    return EC_OK;
}

template <bool G, int B>
int launch_fp8_b(const Fp8Args& a, size_t smem, int grid, int block, cudaStream_t s) {
    if (set_smem(fp8_kernel<G, B>, smem) != EC_OK) return EC_ERR_CUDA;
    return launch_ex(fp8_kernel<G, B>, grid, block, smem, s, a);
}

int launch_fp8(bool gemv, const Fp8Args& a, size_t smem, int grid, int block, cudaStream_t s) {
    if (!gemv) return launch_fp8_b<false, 1>(a, smem, grid, block, s);
    if (a.batch <= 1) return launch_fp8_b<true, 1>(a, smem, grid, block, s);
    if (a.batch <= 2) return launch_fp8_b<true, 2>(a, smem, grid, block, s);
    if (a.batch <= 4) return launch_fp8_b<true, 4>(a, smem, grid, block, s);
    if (a.batch <= 8) return launch_fp8_b<true, 8>(a, smem, grid, block, s);
    return launch_fp8_b<true, 16>(a, smem, grid, block, s);
}

/* FP8 GEMV (y != nullptr) or decode: one CTA per SM with the slot table, the value
 * tables and x in shared memory, two tile buffers per warp; batch rows in passes. */
int fp8_run(const ec_matrix* W, const uint16_t* x, float* y, uint16_t* out, int batch, cudaStream_t s,
            DeviceInfo* d) {
    Fp8Args a{};
    a.m = fp8_desc(W);
    a.m.y = y;
    a.m.out = out;
    a.status = d->status;
    const bool gemv = y != nullptr;
    if (gemv && (a.m.atomic_y || W->hdr.n_tiles == 0)) {
        if (cudaMemsetAsync(y, 0, sizeof(float) * (size_t)batch * (size_t)W->hdr.n_rows, s) != cudaSuccess)
            return EC_ERR_CUDA;
    }
    if (W->hdr.n_tiles == 0) return EC_OK;
    const size_t table = ((size_t)4 << a.m.prob_bits) + 4 * EC_FP8_VALUE_WORDS;
    const size_t per_warp = 2 * rans_buf_bytes(a.m.words_cap);
    const int64_t kp = W->hdr.k_pad, K = W->hdr.k_cols;
    const size_t xrow = gemv ? (size_t)2 * kp : 0;
    if (table + xrow + 4 * per_warp > d->smem_optin) return EC_ERR_UNSUPPORTED;
    const int cap = gemv ? rans_max_warps(batch <= 1 ? 1 : batch <= 2 ? 2 : batch <= 4 ? 4 : batch <= 8 ? 8 : 16)
                         : rans_max_warps(1);
    const int warps = (int)std::min<size_t>(cap, (d->smem_optin - table - xrow) / per_warp);
    const size_t fixed = table + (size_t)warps * per_warp;
    const int per_pass = gemv ? (int)std::min<size_t>(std::min(batch, kFmaMaxRows), (d->smem_optin - fixed) / xrow) : 1;
    if (per_pass < 1) return EC_ERR_UNSUPPORTED;
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(d->sms, (W->hdr.n_tiles + warps - 1) / warps));
    const int passes = gemv ? batch : 1;
    for (int b0 = 0; b0 < passes; b0 += per_pass) {
        const int nb = gemv ? std::min(per_pass, batch - b0) : 0;
        a.batch = nb;
        a.x = gemv ? x + (int64_t)b0 * K : nullptr;
        if (gemv) a.m.y = y + (int64_t)b0 * W->hdr.n_rows;
        const int rc = launch_fp8(gemv, a, fixed + xrow * nb, grid, warps * 32, s);
        if (rc != EC_OK) return rc;
    }
    return EC_OK;
}

template <bool G, int B, bool P>
int launch_exp_b(const ExpArgs& a, size_t smem, int grid, int block, cudaStream_t s) {
    if (set_smem(exp_kernel<G, B, P>, smem) != EC_OK) return EC_ERR_CUDA;
    return launch_ex(exp_kernel<G, B, P>, grid, block, smem, s, a);
}

template <bool P>
int launch_exp_p(bool gemv, const ExpArgs& a, size_t smem, int grid, int block, cudaStream_t s) {
    if (!gemv) return launch_exp_b<false, 1, P>(a, smem, grid, block, s);
    if (a.batch <= 1) return launch_exp_b<true, 1, P>(a, smem, grid, block, s);
    if (a.batch <= 2) return launch_exp_b<true, 2, P>(a, smem, grid, block, s);
    if (a.batch <= 4) return launch_exp_b<true, 4, P>(a, smem, grid, block, s);
    if (a.batch <= 8) return launch_exp_b<true, 8, P>(a, smem, grid, block, s);
    return launch_exp_b<true, 16, P>(a, smem, grid, block, s);
}

/* Exponent-coded GEMV (y != nullptr) or decode: one CTA per SM with the slot table,
 * the exponent pairs and x in shared memory, two tile buffers per warp; batch rows in
 * passes. */
int exp_run(const ec_matrix* W, const uint16_t* x, float* y, uint16_t* out, int batch, cudaStream_t s,
            DeviceInfo* d) {
    ExpArgs a{};
    a.m = exp_desc(W);
    a.m.y = y;
    a.m.out = out;
    a.status = d->status;
    const bool gemv = y != nullptr;
    if (gemv && (a.m.atomic_y || W->hdr.n_tiles == 0)) {
        if (cudaMemsetAsync(y, 0, sizeof(float) * (size_t)batch * (size_t)W->hdr.n_rows, s) != cudaSuccess)
            return EC_ERR_CUDA;
    }
    if (W->hdr.n_tiles == 0) return EC_OK;
    const size_t table = ((size_t)4 << a.m.prob_bits) + 1024;
    const size_t per_warp = 2 * rans_buf_bytes(a.m.words_cap);
    const int64_t kp = W->hdr.k_pad, K = W->hdr.k_cols;
    const size_t xrow = gemv ? (size_t)2 * kp : 0;
    if (table + xrow + 4 * per_warp > d->smem_optin) return EC_ERR_UNSUPPORTED;
    const int cap = gemv ? rans_max_warps(batch <= 1 ? 1 : batch <= 2 ? 2 : batch <= 4 ? 4 : batch <= 8 ? 8 : 16)
                         : rans_max_warps(1);
    const int warps = (int)std::min<size_t>(cap, (d->smem_optin - table - xrow) / per_warp);
    const size_t fixed = table + (size_t)warps * per_warp;
    const int per_pass = gemv ? (int)std::min<size_t>(std::min(batch, kFmaMaxRows), (d->smem_optin - fixed) / xrow) : 1;
    if (per_pass < 1) return EC_ERR_UNSUPPORTED;
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(d->sms, (W->hdr.n_tiles + warps - 1) / warps));
    const int passes = gemv ? batch : 1;
    for (int b0 = 0; b0 < passes; b0 += per_pass) {
        const int nb = gemv ? std::min(per_pass, batch - b0) : 0;
        a.batch = nb;
        a.x = gemv ? x + (int64_t)b0 * K : nullptr;
        if (gemv) a.m.y = y + (int64_t)b0 * W->hdr.n_rows;
        const size_t sm = fixed + xrow * nb;
        const int rc = a.m.tuple == 2 ? launch_exp_p<true>(gemv, a, sm, grid, warps * 32, s)
                                      : launch_exp_p<false>(gemv, a, sm, grid, warps * 32, s);
        if (rc != EC_OK) return rc;
    }
    return EC_OK;
}
/* ---- not in the Huffman GEMV: end ---- */

/* ---- E8 decode: begin ---- */
/* E8 decode: one CTA per SM, the 17 tables in shared memory, two tile buffers per warp. */
/* Warps per CTA and tile buffers per warp.  Two buffers when 32 warps fit with
 * them, else one buffer and as many warps as fit (an issue-bound decode keeps the SM
 * busy with the other warps while one waits for its next tile).  The warp count is
 * then lowered to the fewest that keep the same number of tile rounds, so that the
 * last round is full. */
struct E8Plan {
    int warps, nbuf;
};
E8Plan e8_plan(size_t tables, size_t buf, int64_t n_tiles, const DeviceInfo* d) {
    const size_t room = d->smem_optin - tables;
    int nbuf = room / (2 * buf) >= (size_t)kMaxHW ? 2 : 1;
    int wmax = (int)std::min<size_t>(kMaxHW, room / (nbuf * buf));
    if (wmax < 1) {
        nbuf = 1;
        wmax = (int)std::min<size_t>(kMaxHW, room / buf);
    }
    const int64_t per_sm = (n_tiles + d->sms - 1) / d->sms;
    const int64_t rounds = std::max<int64_t>(1, (per_sm + wmax - 1) / wmax);
    const int warps = (int)std::max<int64_t>(1, std::min<int64_t>(wmax, (per_sm + rounds - 1) / rounds));
    return {warps, nbuf};
}

template <int PB, int OUT>
int e8_launch(E8Args a, int64_t n_tiles, cudaStream_t s, DeviceInfo* d) {
    const size_t tables = e8_table_bytes(PB), buf = rans_buf_bytes(a.m.words_cap);
    if (tables + buf + kE8Guard > d->smem_optin) return EC_ERR_UNSUPPORTED; /* not for tiles of <= 1024 vectors */
    const E8Plan p = e8_plan(tables + kE8Guard, buf, n_tiles, d);
    a.nbuf = p.nbuf;
    const size_t smem = tables + (size_t)(p.warps * p.nbuf) * buf + kE8Guard;
    if (set_smem(e8_kernel<PB, OUT>, smem) != EC_OK) return EC_ERR_CUDA;
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(d->sms, (n_tiles + p.warps - 1) / p.warps));
    return launch_ex(e8_kernel<PB, OUT>, grid, p.warps * 32, smem, s, a);
}

template <int OUT>
int e8_launch_pb(const E8Args& a, int64_t nt, cudaStream_t s, DeviceInfo* d) {
    switch (a.m.prob_bits) {
        case 9: return e8_launch<9, OUT>(a, nt, s, d);
        case 10: return e8_launch<10, OUT>(a, nt, s, d);
        case 11: return e8_launch<11, OUT>(a, nt, s, d);
        case 12: return e8_launch<12, OUT>(a, nt, s, d);
        default: return EC_ERR_CORRUPT;
    }
}

int e8_run(const ec_matrix* W, void* out, int dtype, cudaStream_t s, DeviceInfo* d) {
    E8Args a{};
    a.m = e8_desc(W);
    a.m.out = out;
    a.status = d->status;
    const int64_t nt = W->hdr.n_tiles;
    if (nt == 0) return EC_OK;
    switch (dtype) {
        case EC_DTYPE_BF16: return e8_launch_pb<0>(a, nt, s, d);
        case EC_DTYPE_FP8_E4M3: return e8_launch_pb<1>(a, nt, s, d);
        case EC_DTYPE_INT8: return e8_launch_pb<2>(a, nt, s, d);
        default: return EC_ERR_INVALID_ARG;
    }
}
/* ---- E8 decode: end ---- */

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


/* ---- not in the Huffman GEMV: begin ---- */
/* ------------------------------------------------------------ prefill GEMM */
/* The Huffman decode kernel over a.total_tiles tiles (a.m, a.count, a.sub_words set). */
int launch_huff_decode(HuffDecodeArgs& a, int code_bytes, bool lng, cudaStream_t stream, DeviceInfo* d) {
    code_bytes = (code_bytes + 15) & ~15;
    a.status = d->status;
    a.code_bytes = code_bytes;
    const size_t per_warp = huff_warp_bytes(code_bytes), fixed = kPairTabBytes + 4 * (size_t)a.sub_words;
    if (fixed + 4 * per_warp > d->smem_optin) return EC_ERR_UNSUPPORTED;
    const int warps = (int)std::min<size_t>(kDecodeWarps, (d->smem_optin - fixed) / per_warp);
    const size_t smem = fixed + (size_t)warps * per_warp;
    auto kern = lng ? huff_decode_kernel<true> : huff_decode_kernel<false>;
    if (set_smem(kern, smem) != EC_OK) return EC_ERR_CUDA;
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(d->sms, (a.total_tiles + warps - 1) / warps));
    return launch_ex(kern, grid, warps * 32, smem, stream, a);
}

/* Rows [rows, cols] BF16 with row stride ld elements as TMA boxes of 64 columns x
 * box_rows rows with the 128-byte swizzle of the MMA operands; columns past `cols`
 * and rows past `rows` read as zero.  ld % 8 == 0 and p 16-byte aligned. */
int encode_rows_map(CUtensorMap* map, const uint16_t* p, int64_t cols, int64_t rows, int64_t ld, int box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return EC_ERR_CUDA;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)box_rows}, estr[2] = {1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (void*)p, dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? EC_OK : EC_ERR_CUDA;
}

struct GemmPlan {
    int bn, n_tiles, m_tiles, kblocks, ksplit, kbps, stages, grid;
    uint32_t tmem_cols;
    size_t smem, part_bytes;
};

/* Tiles of 128 rows x bn batch rows (batch split evenly into tiles of at most 256);
 * K split so that about one work item per SM exists (at least 4 blocks of 64
 * columns per split), within part_cap bytes of partial sums. */
GemmPlan plan_gemm(int64_t rows, int64_t K, int batch, int sms, size_t smem_optin, size_t part_cap) {
    GemmPlan p{};
    p.n_tiles = (batch + 255) / 256;
    const int per = (batch + p.n_tiles - 1) / p.n_tiles;
    p.bn = (per + 15) & ~15;
    p.m_tiles = (int)((rows + kGemmBM - 1) / kGemmBM);
    p.kblocks = (int)std::max<int64_t>(1, (K + kGemmBK - 1) / kGemmBK);
    const int64_t tiles = (int64_t)p.m_tiles * p.n_tiles;
    int ks = (int)std::max<int64_t>(1, std::min<int64_t>(sms / std::max<int64_t>(1, tiles), p.kblocks / 4));
    for (; ks > 1; --ks) {
        const int kbps = (p.kblocks + ks - 1) / ks, n = (p.kblocks + kbps - 1) / kbps;
        if ((size_t)n * (size_t)batch * (size_t)rows * 4 <= part_cap) break;
    }
    p.kbps = (p.kblocks + ks - 1) / ks;
    p.ksplit = (p.kblocks + p.kbps - 1) / p.kbps;
    p.part_bytes = p.ksplit > 1 ? (size_t)p.ksplit * (size_t)batch * (size_t)rows * 4 : 0;
    const size_t stage = kGemmABytes + (size_t)p.bn * 128, extra = 64;
    p.stages = (int)std::min<size_t>(8, (smem_optin - extra) / (stage + 16));
    p.smem = (size_t)p.stages * (stage + 16) + extra;
    p.tmem_cols = 32;
    while (p.tmem_cols < 2u * (uint32_t)p.bn) p.tmem_cols <<= 1;
    p.grid = (int)std::min<int64_t>(sms, tiles * p.ksplit);
    return p;
}

/* y[b * ldy + row_off + r] = sum_k A[r][k] x[b][k] for the rows r < rows of A (ld
 * elements apart) and batch rows b of x (xld apart): the tensor-core kernel, then
 * the split reduction when K is split (partial sums in part, part_cap bytes). */
int gemm_run(const uint16_t* A, int64_t rows, int64_t K, int64_t lda, const uint16_t* x, int64_t xld, int batch,
             float* y, int64_t ldy, int64_t row_off, float* part, size_t part_cap, cudaStream_t s, DeviceInfo* d) {
    if (rows == 0 || batch == 0) return EC_OK;
    const GemmPlan p = plan_gemm(rows, K, batch, d->sms, d->smem_optin, part ? part_cap : 0);
    if (p.stages < 2) return EC_ERR_UNSUPPORTED;
    if (rows > INT32_MAX || (int64_t)p.m_tiles * p.n_tiles * p.ksplit > INT32_MAX) return EC_ERR_UNSUPPORTED;
    GemmArgs a{};
    int rc = encode_rows_map(&a.amap, A, K, rows, lda, kGemmBM);
    if (rc == EC_OK) rc = encode_rows_map(&a.bmap, x, K, batch, xld, p.bn);
    if (rc != EC_OK) return rc;
    a.y = y;
    a.part = part;
    a.ldy = ldy;
    a.row_off = row_off;
    a.rows = (int)rows;
    a.batch = batch;
    a.kblocks = p.kblocks;
    a.bn = p.bn;
    a.m_tiles = p.m_tiles;
    a.n_tiles = p.n_tiles;
    a.ksplit = p.ksplit;
    a.kb_per_split = p.kbps;
    a.stages = p.stages;
    /* kind::f16: FP32 accumulators, BF16 A and B, both K-major, N >> 3, M >> 4 */
    a.idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(p.bn >> 3) << 17) | ((uint32_t)(kGemmBM >> 4) << 24);
    a.tmem_cols = p.tmem_cols;
    a.status = d->status;
    if (set_smem(gemm_bf16_kernel, p.smem) != EC_OK) return EC_ERR_CUDA;
    if ((rc = launch_ex(gemm_bf16_kernel, p.grid, kGemmThreads, p.smem, s, a)) != EC_OK) return rc;
    if (p.ksplit > 1) {
        const int64_t n = (int64_t)batch * rows;
        const int grid = (int)std::min<int64_t>((n + 255) / 256, 8 * (int64_t)d->sms);
        rc = launch_ex(gemm_reduce_kernel, grid, 256, 0, s, (const float*)part, p.ksplit, batch, (int)rows, y, ldy,
                       row_off);
    }
    return rc;
}

/* How the prefill GEMM of W at `batch` rows uses its work buffer: chunks of
 * chunk_rows decoded rows (row stride ld) at offset 0, x with row stride ld at
 * x_off when K % 8 != 0 (TMA rows must be 16-byte aligned), partial sums at
 * part_off (part_cap bytes). */
struct PrefillPlan {
    int64_t ld, chunk_rows;
    size_t x_off, part_off, part_cap, need;
};

constexpr size_t kPrefillChunkBytes = size_t(128) << 20; /* decoded rows per chunk (about the L2 size) */

size_t round256(size_t v) { return (v + 255) & ~size_t(255); }

/* Work bytes for chunks of cr rows (0: the partial sums alone would not fit). */
size_t prefill_need(const ec_matrix* W, int batch, int64_t cr, int64_t ld, const DeviceInfo& d, size_t* x_off,
                    size_t* part_off, size_t* part_cap) {
    const ec_blob_header& h = W->hdr;
    const size_t chunk = round256((size_t)cr * (size_t)ld * 2);
    const size_t xb = h.k_cols % 8 ? round256((size_t)batch * (size_t)ld * 2) : 0;
    /* the partial sums of the largest plan among the full and the last chunk */
    const int64_t last = h.n_rows % cr ? h.n_rows % cr : cr;
    size_t part = 0;
    for (int64_t r : {cr, last}) part = std::max(part, plan_gemm(r, h.k_cols, batch, d.sms, d.smem_optin, SIZE_MAX).part_bytes);
    *x_off = chunk;
    *part_off = chunk + xb;
    *part_cap = part;
    return chunk + xb + part;
}

/* Warps per CTA that the Huffman decode kernel launches with for W. */
int huff_decode_warps(const ec_matrix* W, const DeviceInfo& d) {
    const int code_bytes = (std::max(16, staged_code_bytes(W)) + 15) & ~15;
    const bool sub = huff_hier(W) && W->hdr.huff_sub_tables > 0 && W->hdr.huff_sub_tables <= kSubSmemTables;
    const size_t per_warp = huff_warp_bytes(code_bytes), fixed = kPairTabBytes + (sub ? 1024 * (size_t)W->hdr.huff_sub_tables : 0);
    if (fixed + per_warp > d.smem_optin) return 1;
    return (int)std::max<size_t>(1, std::min<size_t>(kDecodeWarps, (d.smem_optin - fixed) / per_warp));
}

/* Rows per chunk: a multiple of `step` (chunk starts fall on tile starts), the
 * most that fit in work_bytes (0: the default chunk size).  By default a chunk holds the tiles of whole rounds of the decode
 * launch (one tile per warp of every CTA), as many rounds as fit in about
 * kPrefillChunkBytes (at least one): a chunk of 1.3 rounds would take as long to
 * decode as one of 2. */
int plan_prefill(const ec_matrix* W, int batch, size_t work_bytes, const DeviceInfo& d, PrefillPlan* pp) {
    const ec_blob_header& h = W->hdr;
    pp->ld = (h.k_cols + 7) & ~int64_t(7);
    int64_t step = h.n_rows, cr = h.n_rows;
    if (W->kind == EC_KIND_HUFFMAN_BF16 && h.k_pad > 0) {
        const int64_t T = 32 * (int64_t)h.steps;
        step = T / std::gcd(T, h.k_pad);
        const int64_t slots = (int64_t)d.sms * huff_decode_warps(W, d);
        const int64_t round_bytes = slots * T * 2;
        const int64_t rounds = std::max<int64_t>(1, (int64_t)kPrefillChunkBytes / std::max<int64_t>(1, round_bytes));
        cr = rounds * slots * T / h.k_pad;
    }
    step = std::max<int64_t>(1, std::min(step, h.n_rows));
    cr = std::max(step, cr / step * step);
    cr = std::min(cr, h.n_rows);
    for (;;) {
        const size_t need = prefill_need(W, batch, cr, pp->ld, d, &pp->x_off, &pp->part_off, &pp->part_cap);
        if (work_bytes == 0 || need <= work_bytes) {
            pp->chunk_rows = cr;
            pp->need = need;
            return EC_OK;
        }
        if (cr <= step) return EC_ERR_INVALID_ARG; /* the work buffer is too small */
        cr = std::max(step, (cr - 1) / step * step);
    }
}

/* ---- not in the Huffman GEMV: end ---- */
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
    if (Ws[0]->kind == EC_KIND_E8) return EC_ERR_UNSUPPORTED; /* decoded to a dense matrix instead */
    if (Ws[0]->kind == EC_KIND_HUFFMAN_BF16) return huff_gemv(Ws, count, x, ys, batch, stream, dev, d);
    for (int k = 0; k < count; ++k) {
        rc = Ws[0]->kind == EC_KIND_RANS_FP8   ? fp8_run(Ws[k], x, ys[k], nullptr, batch, stream, d)
             : Ws[0]->kind == EC_KIND_RANS_EXP ? exp_run(Ws[k], x, ys[k], nullptr, batch, stream, d)
                                              : rans_run(Ws[k], x, ys[k], nullptr, batch, stream, d);
        if (rc != EC_OK) return rc;
    }
    return EC_OK;
}

extern "C" int ec_gemv_path(const ec_matrix* const* Ws, int count, int batch) {
    if (!Ws || count < 1 || count > EC_MAX_GROUP) return EC_ERR_INVALID_ARG;
    if (batch < 1 || batch > EC_MAX_BATCH) return batch < 1 ? EC_ERR_INVALID_ARG : EC_ERR_UNSUPPORTED;
    for (int k = 0; k < count; ++k) {
        if (!Ws[k]) return EC_ERR_INVALID_ARG;
        if (Ws[k]->kind != Ws[0]->kind || Ws[k]->hdr.k_cols != Ws[0]->hdr.k_cols) return EC_ERR_SHAPE;
    }
    if (Ws[0]->kind == EC_KIND_E8) return EC_ERR_UNSUPPORTED;
    return Ws[0]->kind == EC_KIND_HUFFMAN_BF16 && use_mma(Ws, count, batch) ? EC_PATH_TENSOR_CORES : EC_PATH_CUDA_CORES;
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
    bool lng = false;
    for (int k = 0; k < count; ++k) {
        if ((rc = check_matrix(Ws[k], dev)) != EC_OK) return rc;
        const int64_t n = Ws[k]->hdr.n_rows * Ws[k]->hdr.k_cols;
        if (n > 0 && (!outs[k] || !aligned16(outs[k]))) return EC_ERR_INVALID_ARG;
        if (Ws[k]->kind == EC_KIND_RANS_INT4) {
            if ((rc = rans_run(Ws[k], nullptr, nullptr, outs[k], 1, stream, d)) != EC_OK) return rc;
            continue;
        }
        if (Ws[k]->kind == EC_KIND_RANS_EXP) {
            if ((rc = exp_run(Ws[k], nullptr, nullptr, outs[k], 1, stream, d)) != EC_OK) return rc;
            continue;
        }
        if (Ws[k]->kind == EC_KIND_RANS_FP8) {
            if ((rc = fp8_run(Ws[k], nullptr, nullptr, outs[k], 1, stream, d)) != EC_OK) return rc;
            continue;
        }
        if (Ws[k]->kind == EC_KIND_E8) {
            if ((rc = e8_run(Ws[k], outs[k], EC_DTYPE_BF16, stream, d)) != EC_OK) return rc;
            continue;
        }
        HuffMat m = huff_desc(Ws[k]);
        m.out = outs[k];
        m.tile_begin = total;
        total += Ws[k]->hdr.n_tiles;
        code_bytes = std::max(code_bytes, staged_code_bytes(Ws[k]));
        lng = lng || huff_hier(Ws[k]);
        /* one matrix at a time is resident: its sub-tables are staged when they fit */
        if (huff_hier(Ws[k]) && m.n_sub > 0 && m.n_sub <= kSubSmemTables) {
            m.sub_smem = 0;
            a.sub_words = std::max(a.sub_words, 256 * m.n_sub);
        }
        a.m[a.count++] = m;
    }
    if (a.count == 0 || total == 0) return EC_OK;
    a.total_tiles = total;
    return launch_huff_decode(a, code_bytes, lng, stream, d);
}

/* ---- not in the Huffman GEMV: begin ---- */
extern "C" int ec_gemm_work_bytes(const ec_matrix* W, int batch, size_t* bytes) {
    if (!W || !bytes || batch < 1) return EC_ERR_INVALID_ARG;
    int dev = 0;
    if (current_device(&dev) != EC_OK) return EC_ERR_CUDA;
    DeviceInfo* d = nullptr;
    int rc = device_info(dev, &d);
    if (rc != EC_OK) return rc;
    PrefillPlan pp;
    if ((rc = plan_prefill(W, batch, 0, *d, &pp)) != EC_OK) return rc;
    *bytes = pp.need;
    return EC_OK;
}

extern "C" int ec_gemm(const ec_matrix* W, const uint16_t* x, float* y, int batch, void* work, size_t work_bytes,
                       cudaStream_t stream) {
    if (!W || !W->d_blob || batch < 1) return EC_ERR_INVALID_ARG;
    int dev = 0;
    if (current_device(&dev) != EC_OK) return EC_ERR_CUDA;
    DeviceInfo* d = nullptr;
    int rc = device_info(dev, &d);
    if (rc != EC_OK) return rc;
    if ((rc = check_matrix(W, dev)) != EC_OK) return rc;
    const ec_blob_header& h = W->hdr;
    const int64_t K = h.k_cols;
    if (!y || !aligned16(y) || (K > 0 && (!x || !aligned16(x)))) return EC_ERR_INVALID_ARG;
    if (h.n_rows == 0) return EC_OK;
    if (K == 0)
        return cudaMemsetAsync(y, 0, sizeof(float) * (size_t)batch * (size_t)h.n_rows, stream) == cudaSuccess
                   ? EC_OK
                   : EC_ERR_CUDA;
    const bool huff = W->kind == EC_KIND_HUFFMAN_BF16;
    if (!huff && K % 8) return EC_ERR_UNSUPPORTED; /* decoded whole, rows K apart: TMA needs 16-byte rows */
    PrefillPlan pp;
    if ((rc = plan_prefill(W, batch, work_bytes, *d, &pp)) != EC_OK) return rc;
    if (!work || !aligned16(work) || work_bytes < pp.need) return EC_ERR_INVALID_ARG;
    uint8_t* wb = (uint8_t*)work;
    uint16_t* chunk = (uint16_t*)wb;
    float* part = pp.part_cap ? (float*)(wb + pp.part_off) : nullptr;
    const uint16_t* xs = x;
    int64_t xld = K;
    if (K % 8) { /* x rows re-strided to ld for TMA (the columns past K are never read) */
        uint16_t* xp = (uint16_t*)(wb + pp.x_off);
        if (cudaMemcpy2DAsync(xp, (size_t)pp.ld * 2, x, (size_t)K * 2, (size_t)K * 2, (size_t)batch,
                              cudaMemcpyDeviceToDevice, stream) != cudaSuccess)
            return EC_ERR_CUDA;
        xs = xp;
        xld = pp.ld;
    }
    if (!huff) { /* one chunk: the whole matrix through its own decoder */
        rc = W->kind == EC_KIND_RANS_INT4  ? rans_run(W, nullptr, nullptr, chunk, 1, stream, d)
             : W->kind == EC_KIND_RANS_FP8 ? fp8_run(W, nullptr, nullptr, chunk, 1, stream, d)
             : W->kind == EC_KIND_RANS_EXP ? exp_run(W, nullptr, nullptr, chunk, 1, stream, d)
                                           : e8_run(W, chunk, EC_DTYPE_BF16, stream, d);
        if (rc != EC_OK) return rc;
        return gemm_run(chunk, h.n_rows, K, K, xs, xld, batch, y, h.n_rows, 0, part, pp.part_cap, stream, d);
    }
    HuffDecodeArgs a{};
    a.count = 1;
    HuffMat m = huff_desc(W);
    m.out = chunk;
    m.out_ld = pp.ld;
    const bool lng = huff_hier(W);
    if (lng && m.n_sub > 0 && m.n_sub <= kSubSmemTables) {
        m.sub_smem = 0;
        a.sub_words = 256 * m.n_sub;
    }
    const int code_bytes = std::max(16, staged_code_bytes(W));
    const int64_t T = 32 * (int64_t)h.steps;
    for (int64_t r0 = 0; r0 < h.n_rows; r0 += pp.chunk_rows) {
        const int64_t r1 = std::min(h.n_rows, r0 + pp.chunk_rows);
        /* chunk starts are tile starts: the chunk's tiles cover exactly its rows */
        const int64_t t0 = r0 * h.k_pad / T, t1 = r1 == h.n_rows ? h.n_tiles : r1 * h.k_pad / T;
        a.m[0] = m;
        a.m[0].out_row0 = r0;
        a.m[0].tile_begin = -t0;
        a.total_tiles = t1 - t0;
        if ((rc = launch_huff_decode(a, code_bytes, lng, stream, d)) != EC_OK) return rc;
        if ((rc = gemm_run(chunk, r1 - r0, K, pp.ld, xs, xld, batch, y, h.n_rows, r0, part, pp.part_cap, stream, d)) !=
            EC_OK)
            return rc;
    }
    return EC_OK;
}

namespace {
/* Whether ec_gemm_group packs W with others into one decode launch. */
bool gemm_packable(const ec_matrix* W) { return W->kind == EC_KIND_HUFFMAN_BF16 && W->hdr.k_cols % 8 == 0; }

/* Partial-sum bytes the GEMM of a whole packable matrix needs at `batch`. */
size_t gemm_part_bytes(const ec_matrix* W, int batch, const DeviceInfo& d) {
    return plan_gemm(W->hdr.n_rows, W->hdr.k_cols, batch, d.sms, d.smem_optin, SIZE_MAX).part_bytes;
}
}  // namespace

extern "C" int ec_gemm_group_work_bytes(const ec_matrix* const* Ws, int count, int batch, size_t* bytes) {
    if (!Ws || !bytes || count < 1 || count > kMaxDecodeBatch || batch < 1) return EC_ERR_INVALID_ARG;
    int dev = 0;
    if (current_device(&dev) != EC_OK) return EC_ERR_CUDA;
    DeviceInfo* d = nullptr;
    int rc = device_info(dev, &d);
    if (rc != EC_OK) return rc;
    size_t packed = 0, part = 0, alone = 0;
    for (int k = 0; k < count; ++k) {
        if (!Ws[k]) return EC_ERR_INVALID_ARG;
        if (gemm_packable(Ws[k])) {
            packed += round256((size_t)Ws[k]->hdr.n_rows * (size_t)Ws[k]->hdr.k_cols * 2);
            part = std::max(part, round256(gemm_part_bytes(Ws[k], batch, *d)));
        } else {
            PrefillPlan pp;
            if ((rc = plan_prefill(Ws[k], batch, 0, *d, &pp)) != EC_OK) return rc;
            alone = std::max(alone, pp.need);
        }
    }
    *bytes = std::max(packed + part, alone);
    return EC_OK;
}

extern "C" int ec_gemm_group(const ec_matrix* const* Ws, int count, const uint16_t* const* xs, float* const* ys,
                             int batch, void* work, size_t work_bytes, cudaStream_t stream) {
    if (!Ws || !xs || !ys || count < 1 || count > kMaxDecodeBatch || batch < 1) return EC_ERR_INVALID_ARG;
    if (!work || !aligned16(work)) return EC_ERR_INVALID_ARG;
    int dev = 0;
    if (current_device(&dev) != EC_OK) return EC_ERR_CUDA;
    DeviceInfo* d = nullptr;
    int rc = device_info(dev, &d);
    if (rc != EC_OK) return rc;
    size_t part = 0;
    for (int k = 0; k < count; ++k) {
        if (!Ws[k] || !Ws[k]->d_blob) return EC_ERR_INVALID_ARG;
        if ((rc = check_matrix(Ws[k], dev)) != EC_OK) return rc;
        if (!ys[k] || !aligned16(ys[k]) || (Ws[k]->hdr.k_cols > 0 && (!xs[k] || !aligned16(xs[k]))))
            return EC_ERR_INVALID_ARG;
        if (gemm_packable(Ws[k])) part = std::max(part, round256(gemm_part_bytes(Ws[k], batch, *d)));
    }
    /* [decoded matrices of one pack | partial sums] */
    const size_t area = work_bytes > part ? work_bytes - part : 0;
    float* part_p = part ? (float*)((uint8_t*)work + area) : nullptr;
    std::vector<int> pack;
    size_t used = 0;
    auto flush = [&]() -> int {
        if (pack.empty()) return EC_OK;
        HuffDecodeArgs a{};
        int64_t total = 0;
        int code_bytes = 16;
        bool lng = false;
        size_t off = 0;
        std::vector<size_t> at;
        for (int k : pack) {
            const ec_matrix* W = Ws[k];
            HuffMat m = huff_desc(W);
            m.out = (uint16_t*)((uint8_t*)work + off);
            m.tile_begin = total;
            at.push_back(off);
            off += round256((size_t)W->hdr.n_rows * (size_t)W->hdr.k_cols * 2);
            total += W->hdr.n_tiles;
            code_bytes = std::max(code_bytes, staged_code_bytes(W));
            lng = lng || huff_hier(W);
            if (huff_hier(W) && m.n_sub > 0 && m.n_sub <= kSubSmemTables) { /* one matrix at a time is resident */
                m.sub_smem = 0;
                a.sub_words = std::max(a.sub_words, 256 * m.n_sub);
            }
            a.m[a.count++] = m;
        }
        int r = EC_OK;
        if (total > 0) {
            a.total_tiles = total;
            if ((r = launch_huff_decode(a, code_bytes, lng, stream, d)) != EC_OK) return r;
        }
        for (size_t i = 0; i < pack.size(); ++i) {
            const ec_matrix* W = Ws[pack[i]];
            const ec_blob_header& h = W->hdr;
            if (h.n_rows == 0) continue;
            if (h.k_cols == 0) {
                if (cudaMemsetAsync(ys[pack[i]], 0, sizeof(float) * (size_t)batch * (size_t)h.n_rows, stream) !=
                    cudaSuccess)
                    return EC_ERR_CUDA;
                continue;
            }
            const uint16_t* rows = (const uint16_t*)((uint8_t*)work + at[i]);
            if ((r = gemm_run(rows, h.n_rows, h.k_cols, h.k_cols, xs[pack[i]], h.k_cols, batch, ys[pack[i]], h.n_rows,
                              0, part_p, part, stream, d)) != EC_OK)
                return r;
        }
        pack.clear();
        used = 0;
        return EC_OK;
    };
    for (int k = 0; k < count; ++k) {
        const ec_matrix* W = Ws[k];
        const size_t sz = gemm_packable(W) ? round256((size_t)W->hdr.n_rows * (size_t)W->hdr.k_cols * 2) : SIZE_MAX;
        if (sz <= area) {
            if (used + sz > area && (rc = flush()) != EC_OK) return rc;
            pack.push_back(k);
            used += sz;
            continue;
        }
        /* alone, in row chunks of its own */
        if ((rc = flush()) != EC_OK) return rc;
        if ((rc = ec_gemm(W, xs[k], ys[k], batch, work, work_bytes, stream)) != EC_OK) return rc;
    }
    return flush();
}

extern "C" int ec_bf16_gemm(const uint16_t* w, int64_t n_rows, int64_t k_cols, const uint16_t* x, float* y, int batch,
                            void* work, size_t work_bytes, cudaStream_t stream) {
    if (n_rows < 0 || k_cols < 0 || batch < 1) return EC_ERR_INVALID_ARG;
    if (n_rows == 0) return EC_OK;
    if (!y || !aligned16(y)) return EC_ERR_INVALID_ARG;
    if (k_cols == 0)
        return cudaMemsetAsync(y, 0, sizeof(float) * (size_t)batch * (size_t)n_rows, stream) == cudaSuccess
                   ? EC_OK
                   : EC_ERR_CUDA;
    if (!w || !x || !aligned16(w) || !aligned16(x)) return EC_ERR_INVALID_ARG;
    if (k_cols % 8) return EC_ERR_UNSUPPORTED;
    if (work && !aligned16(work)) return EC_ERR_INVALID_ARG;
    int dev = 0;
    if (current_device(&dev) != EC_OK) return EC_ERR_CUDA;
    DeviceInfo* d = nullptr;
    int rc = device_info(dev, &d);
    if (rc != EC_OK) return rc;
    return gemm_run(w, n_rows, k_cols, k_cols, x, k_cols, batch, y, n_rows, 0, (float*)work, work ? work_bytes : 0,
                    stream, d);
}
/* ---- not in the Huffman GEMV: end ---- */

extern "C" int ec_decode(const ec_matrix* W, uint16_t* out, cudaStream_t stream) {
    return ec_decode_batch(&W, &out, 1, stream);
}

extern "C" int ec_decode_as(const ec_matrix* W, void* out, int dtype, cudaStream_t stream) {
    if (!W || !W->d_blob) return EC_ERR_INVALID_ARG;
    if (dtype != EC_DTYPE_BF16 && dtype != EC_DTYPE_FP8_E4M3 && dtype != EC_DTYPE_INT8) return EC_ERR_INVALID_ARG;
    if (W->kind != EC_KIND_E8) {
        if (dtype != EC_DTYPE_BF16) return EC_ERR_UNSUPPORTED;
        uint16_t* o = (uint16_t*)out;
        return ec_decode_batch(&W, &o, 1, stream);
    }
    int dev = 0;
    if (current_device(&dev) != EC_OK) return EC_ERR_CUDA;
    DeviceInfo* d = nullptr;
    int rc = device_info(dev, &d);
    if (rc != EC_OK) return rc;
    if ((rc = check_matrix(W, dev)) != EC_OK) return rc;
    if (W->hdr.n_rows * W->hdr.k_cols > 0 && (!out || !aligned16(out))) return EC_ERR_INVALID_ARG;
    return e8_run(W, out, dtype, stream, d);
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
    /* and the status word of the allocation-free GEMV (word 0 of its scratch array;
     * symbol copies allocate nothing) */
    int w = 0;
    if (cudaMemcpyFromSymbol(&w, g_ec_static_scratch, sizeof(int)) != cudaSuccess) return EC_ERR_CUDA;
    if (w) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_ec_static_scratch, &zero, sizeof(int)) != cudaSuccess) return EC_ERR_CUDA;
    }
    return v || w ? EC_ERR_CORRUPT : EC_OK;
}

/* Allocation-free GEMV (declared in ec.h, where its contract is described). */
extern "C" int ec_gemv_static(const ec_matrix* W, const uint16_t* x, float* y, int batch, cudaStream_t stream) {
    if (!W || !W->d_blob) return EC_ERR_INVALID_ARG;
    if (batch < 1) return EC_ERR_INVALID_ARG;
    if (batch > EC_MAX_BATCH || W->kind != EC_KIND_HUFFMAN_BF16) return EC_ERR_UNSUPPORTED;
    if (!y || !aligned16(y) || (W->hdr.k_cols > 0 && (!x || !aligned16(x)))) return EC_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return EC_ERR_CUDA;
    int rc = check_matrix(W, dev);
    if (rc != EC_OK) return rc;
    StaticDevice* d = nullptr;
    if ((rc = static_device(dev, &d)) != EC_OK) return rc;
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
    a.code_bytes = staged_code_bytes(W);
    a.part = d->scratch + kStaticHeaderFloats;
    a.part_slots = (int)slots;
    a.sub_words = plan_sub_tables(a.m, 1);
    if (a.code_bytes < 16) a.code_bytes = 16;
    /* (the status word is not cleared here: a report stays until ec_status reads it) */
    GemvPlan pl;
    DeviceInfo di{};
    di.sms = d->sms;
    di.smem_optin = d->smem_optin;
    if ((rc = plan_huff_gemv(di, 1, a.code_bytes, h.k_pad, batch, h.n_tiles, a.sub_words, &pl)) != EC_OK) return rc;
    set_tile_stride(a.m[0], (int64_t)pl.grid * pl.warps);
    for (int b0 = 0; b0 < batch; b0 += pl.per_pass) {
        const int nb = std::min(pl.per_pass, batch - b0);
        a.batch = nb;
        a.x = x + (int64_t)b0 * h.k_cols;
        if ((rc = launch_huff_gemv<true>(a, huff_hier(W), pl.fixed + pl.xrow * nb, pl.grid, pl.warps * 32,
                                         stream)) != EC_OK)
            return rc;
        const int64_t n = (int64_t)nb * h.n_rows;
        part_reduce_kernel<<<(unsigned)((n + 255) / 256), 256, 0, stream>>>(a.part, a.part_slots, h.n_rows, h.k_pad,
                                                                           T, nb, y + (int64_t)b0 * h.n_rows);
        if ((rc = launch_result()) != EC_OK) return rc;
    }
    return EC_OK;
}
