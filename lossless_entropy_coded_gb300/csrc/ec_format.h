/*
 * ec_format.h -- device layout of an encoded matrix (shared by the host encoder
 * and the CUDA kernels of this library; nothing outside the library uses it).
 *
 * One contiguous device blob per matrix:
 *
 *   [ec_blob_header, 256 B]
 *   [decode table]            Huffman: pair table, then the hierarchical table
 *                             (level 1 + 256-entry sub-tables).
 *                             rANS:    2^prob_bits u32 slot entries.
 *   [group scales]            rANS only: FP16 [n_rows, k_pad / 128].
 *   [tile offsets]            u32 [n_tiles + 1], record start in 16-byte units.
 *   [tile records]            16-byte aligned, variable length.
 *
 * Coded layout of the weights.  The matrix is padded at the end of every row to
 * k_pad columns (a multiple of EC_HUFF_ROW_ALIGN / EC_RANS_ROW_ALIGN) with zero
 * weights, flattened row-major, and cut into tiles of 32 * steps positions (the
 * last tile may be shorter, always a multiple of the row alignment).
 * Huffman tiles: position q = 256 * (i / 8) + 8 * l + i % 8 is symbol i of lane
 * l, so lane l of the decoding warp owns 8 consecutive positions out of every
 * 256 (8 l .. 8 l + 7, 256 + 8 l .. 256 + 8 l + 7, ...).  rANS tiles: position
 * q = 32 * i + l is symbol i of lane l (positions l, l + 32, l + 64, ...).
 *
 * Huffman tile record (DFloat11's EncodedExponent / PackedSignMantissa /
 * per-thread start offsets, re-cut so every lane owns a fixed number of symbols):
 *   u16 lane_start[32]        byte offset of lane l's codewords in the code area
 *   u8  raw[32 * S16]         (sign << 7) | mantissa, lane-transposed in 16-byte
 *                             chunks: chunk j of lane l (bytes (32 j + l) * 16 ..
 *                             + 15) holds lane l's symbols 16 j .. 16 j + 15, so a
 *                             warp reading chunk j reads 512 contiguous bytes;
 *                             S16 = steps rounded up to 16, the tail zero
 *   u32 code[]                the code area: lane 0's codewords, then lane 1's, ...
 *                             each lane starting on a byte boundary; bit b of the
 *                             area is bit 31 - (b % 32) of word b / 32 (MSB first);
 *                             followed by >= 8 zero bytes, padded to 16 bytes.
 *
 * E8 matrices (kind 3): rows padded to k_pad (a multiple of EC_E8_ROW_ALIGN) with
 * zero points, flattened row-major into 8-weight vectors and cut into tiles of
 * 32 * steps vectors; lane l owns the tile's vectors l, l + 32, ...; a vector is
 * nine symbols (coset, z_1..z_7, m).  Tables: 17 x 32 u32 (freq | cum << 16), table
 * t = 0 for the coset and 1 + 8 c + f for field f under coset c, then 17 x 2^b u8
 * slot -> symbol maps.  [group scales] holds the FP32 row scales [n_rows].  Tile
 * records as rANS below.
 *
 * rANS tile record (EntroPack appendix C.3):
 *   u32 state[32]             the decoder's initial states (the encoder's final ones)
 *   u16 word[]                16-bit payload words in decoder order, padded to 16 B.
 */
#ifndef EC_FORMAT_H_
#define EC_FORMAT_H_

#include <stdint.h>

#define EC_BLOB_MAGIC 0x31434345u /* "ECC1" */
#define EC_BLOB_VERSION 8u

#define EC_L1_BITS 12            /* level-1 Huffman window */
#define EC_SUB_BITS 8            /* bits per sub-table level */
#define EC_PAIR_WORDS (1 << EC_L1_BITS) /* u32 words of the pair table */
#define EC_HUFF_ROW_ALIGN 512    /* k_pad multiple for the Huffman layout (16 symbols x 32 lanes) */
#define EC_MMA_WINDOW_ROWS 31     /* rows whose tiles one tensor-core work item stages together */
#define EC_RANS_ROW_ALIGN 128    /* k_pad multiple for the rANS layout (= scale group) */
#define EC_E8_ROW_ALIGN 256      /* k_pad multiple for the E8 layout (32 vectors of 8) */
#define EC_E8_TABLES 17          /* the coset, and 8 fields under each of 2 cosets */
#define EC_E8_ALPHA 32           /* symbols per field: z + 16 (z in -16..15), m + 16 (m in -8..7) */
#define EC_MAX_CODE_LEN 24

/* bytes of the raw sign/mantissa section of a tile with `steps` symbols per lane */
#define EC_RAW_BYTES(steps) (32 * (((steps) + 15) / 16) * 16)

/* Huffman decode tables, in this order inside the table section:
 *
 * 1. pair table, 2^EC_L1_BITS u32 entries indexed by the next EC_L1_BITS bits of
 *    a lane's stream.  Entry layout (fields chosen so that the entry is already
 *    the exponent half of two BF16 weights [w(i+1) | w(i)]):
 *      bits  7..14  exponent of the first codeword in the window
 *      bits 23..30  exponent of the second codeword (pairs only)
 *      bits  0..3   total length of the two codewords when both end inside the
 *                   window, else 0
 *      bits 16..19  length of the first codeword when it ends inside the window,
 *                   else 0 (longer than the window, or no codeword matches)
 *      all other bits 0.
 *    The decoder reads bits 0..3 to advance; 0 sends it to a second lookup for
 *    the second codeword and, when bits 16..19 are 0 too, to table 2.
 * 2. hierarchical table (u32 entries, below): a 2^EC_L1_BITS level-1 table then
 *    256-entry sub-tables (DFloat11 appendix, Fig. 4 / Fig. 14). */
#define EC_PAIR_LEN_MASK 0x0000000Fu
#define EC_PAIR_FIRST_SHIFT 16
#define EC_PAIR_FIELDS 0x7F8F7F8Fu /* every bit a valid entry may set */

/* Huffman table entry (u32):
 *   symbol:  bits 0..15 = exponent << 7 (the BF16 exponent field), bits 16..20 =
 *            total code length, bits 21..31 = 0
 *   pointer: bit 31 = 1, bits 0..15 = sub-table index, bits 16..20 = bits already
 *            consumed before the sub-table
 *   invalid: bit 30 = 1 (a window no codeword matches; only reachable from corrupt
 *            data or the padding of a one-symbol code). */
#define EC_ENT_PTR 0x80000000u
#define EC_ENT_BAD 0x40000000u

/* rANS slot entry (u32), one code per symbol: bits 0..3 = symbol (code + 8),
 * bits 4..15 = slot - cum[s], bits 16..28 = freq[s].
 * Two codes per symbol (symbol = 16 (c0 + 8) + (c1 + 8) for a lane's steps 2m and
 * 2m + 1): bits 0..7 = symbol, bits 8..19 = slot - cum[s], bits 20..31 =
 * freq[s] - 1. */

/* FP8 blob (kind 4): the table section is 2^prob_bits slot entries in the pair
 * layout above (bits 0..7 = symbol = rank of the code in the top-t table, bits
 * 8..19 = slot - cum[s], bits 20..31 = freq[s] - 1), then 256 FP32 values of the
 * symbols (unused ones 0), then 256 FP32 values of all E4M3 codes (the escapes'
 * values); FP32 row scales at scales_off; u32 record offsets per tile at
 * esc_off_off (record index, n_tiles + 1 entries) and the records at
 * esc_records_off (position in the tile | code << 16, ascending positions within a
 * tile); rANS tile records (32 states, u16 words) as for kind 2, last. */
#define EC_FP8_VALUE_WORDS 512

typedef struct {
    uint32_t magic, version;
    int32_t kind;             /* EC_KIND_* */
    int32_t steps;            /* symbols per lane per tile */
    int64_t n_rows, k_cols, k_pad;
    int64_t n_tiles;
    int64_t table_off, table_words;   /* byte offset, u32 count */
    int64_t scales_off;               /* rANS: byte offset of FP16 scales */
    int64_t tile_off_off;             /* byte offset of u32 tile offsets */
    int64_t records_off;              /* byte offset of the first record */
    int64_t blob_bytes;
    int32_t max_code_bytes;           /* Huffman: largest code area of any tile (bytes) */
    int32_t prob_bits;                /* rANS */
    int32_t max_words;                /* rANS: largest payload of any tile (u16 words) */
    int32_t max_len;                  /* Huffman: longest codeword in use */
    int32_t rans_tuple;               /* rANS: codes per symbol, 1 or 2 */
    int32_t window_code_bytes;        /* Huffman, tiles inside rows: the largest sum of (64 + code area)
                                       * over EC_MMA_WINDOW_ROWS consecutive rows' tiles of one tile
                                       * column; 0 when tiles cross rows */
    uint32_t e8_scale_bits;           /* E8: the shared scale s (FP32 bit pattern) */
    int32_t fp8_table_size;           /* FP8: codes in the decoding table (1..256) */
    int64_t esc_off_off;              /* FP8: byte offset of u32 record offsets [n_tiles + 1] */
    int64_t esc_records_off;          /* FP8: byte offset of the u32 correction records */
    int64_t n_escapes;                /* FP8: correction records */
    uint8_t pad[256 - 4 * 4 - 8 * 10 - 4 * 8 - 8 * 3];
} ec_blob_header;

#endif /* EC_FORMAT_H_ */
