/*
 * ec_format.h -- device layout of an encoded matrix (shared by the host encoder
 * and the CUDA kernels of this library; nothing outside the library uses it).
 *
 * One contiguous device blob per matrix:
 *
 *   [ec_blob_header, 256 B]
 *   [decode table]            Huffman: pair table, then (without window records)
 *                             the hierarchical sub-tables (256 entries each).
 *                             rANS:    2^prob_bits u32 slot entries.
 *   [group scales]            rANS only: FP16 [n_rows, k_pad / 128].
 *   [tile offsets]            u32 [n_tiles + 1], record start in 16-byte units.
 *   [correction records]      FP8: u32 record offsets [n_tiles + 1], then the u32
 *                             records.
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
 *   u16 lane_start[32]        byte offset of lane l's codewords in the code area;
 *                             lane 0 starts at 0, and its slot holds the number of
 *                             window records of the tile instead
 *   u8  raw[32 * S16]         sign and mantissa bits, lane-transposed in 16-byte
 *                             chunks: chunk j of lane l (bytes (32 j + l) * 16 ..
 *                             + 15) holds lane l's symbols 16 j .. 16 j + 15, so a
 *                             warp reading chunk j reads 512 contiguous bytes;
 *                             S16 = steps rounded up to 16, the tail zero.  Each
 *                             little-endian u32 r of a chunk holds symbols i .. i + 3
 *                             (i % 4 == 0) with their sign / mantissa bits where a
 *                             BF16 pair keeps them: the bits 0x807F807F of r are
 *                             [w(i+1) | w(i)], those of r rotated right by 8 are
 *                             [w(i+3) | w(i+2)].  Byte by byte:
 *                               byte 0 = sign(i+3) << 7 | mant(i)
 *                               byte 1 = sign(i)   << 7 | mant(i+2)
 *                               byte 2 = sign(i+2) << 7 | mant(i+1)
 *                               byte 3 = sign(i+1) << 7 | mant(i+3)
 *   u32 code[]                the code area: lane 0's codewords, then lane 1's, ...
 *                             each lane starting on a byte boundary, LSB first: bit
 *                             b of the area is bit b % 32 of word b / 32 (bit b % 8
 *                             of byte b / 8), and a codeword's first bit (its most
 *                             significant in the canonical code) comes first;
 *                             followed by >= 8 zero bytes, padded to 16 bytes
 *   u32 rec[n]                the tile's window records (n = lane_start[0]), zero-
 *                             padded to 16 bytes
 * Window records (window_records = 1): the decoder reads two codewords per lookup
 * of a 12-bit window.  Wherever the two codewords of a lane's pair (symbols 2m,
 * 2m + 1) would not both fit in 12 bits, the encoder writes the codeword of the
 * shortest-coded exponent (header field huff_fill) in place of one (or both) and
 * lists the weight in a record of the tile: u32 position in the tile (13 bits) |
 * (sign << 7 | mantissa) << 13 | true exponent << 21, ascending positions, so a
 * record alone gives both the true and the coded weight (MINE section 4,
 * "Escapes", applied to exponent pairs).  The records follow the code area in the
 * tile record, so the copy that stages the code area brings them along (up to the
 * decoder's staging room).  Huffman tiles hold at most 8192 positions (steps <=
 * EC_HUFF_MAX_STEPS).  Without window records every pair that overflows the window, and
 * every codeword longer than 12 bits, is decoded through the hierarchical tables.
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
#define EC_BLOB_VERSION 11u

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
 *    a lane's stream (the first stream bit is bit 0 of the index).  Fields sit
 *    where they cost the decoder nothing: the two exponents already in the BF16
 *    exponent fields of [w(i+1) | w(i)], everything else under the sign and
 *    mantissa bits that the merge with the raw bytes overwrites:
 *      bits  0..3   advance: the total length of the two codewords when both end
 *                   inside the window; else the first codeword's length when it
 *                   ends inside it; else 0
 *      bits  4..6   0 (the decoder adds whole entries to its bit position, whose
 *                   bit 5 then flips exactly when the position crosses a word)
 *      bits  7..14  exponent of the first codeword; for a first codeword longer
 *                   than the window, bits 7..15 are the index of its level-2
 *                   sub-table instead
 *      bits 16..19  length of the first codeword when it ends inside the window,
 *                   else 0
 *      bits 23..30  exponent of the second codeword (complete pairs only)
 *      bit  31      1 when the pair is not complete (second codeword outside the
 *                   window, first codeword longer than it, or no codeword matches)
 * 2. hierarchical sub-tables (only without window records): 256 u32 entries each,
 *    indexed by the next 8 stream bits after the bits already consumed (DFloat11
 *    appendix, Fig. 4 / Fig. 14, behind a 12-bit first level that is the pair
 *    table):
 *      symbol:  bits 0..15 = exponent << 7, bits 16..20 = total code length
 *      pointer: bit 31 = 1, bits 0..15 = sub-table index, bits 16..20 = stream bits
 *               consumed before that sub-table (20)
 *      invalid: bit 30 = 1 (a window no codeword matches). */
#define EC_PAIR_LEN_MASK 0x0000000Fu
#define EC_PAIR_FIRST_SHIFT 16
#define EC_PAIR_OPEN 0x80000000u   /* pair not complete */
#define EC_PAIR_FIELDS 0xFF8FFF8Fu /* every bit a valid entry may set */
#define EC_HUFF_WINDOW_REC 1       /* ec_blob_header.huff_flags: window records in use */
#define EC_HUFF_MAX_STEPS 256      /* symbols per lane in a Huffman tile */
#define EC_HREC_POS_MASK 0x1FFFu   /* window record: position in the tile */
#define EC_HREC_SM_SHIFT 13        /* window record: sign << 7 | mantissa */
#define EC_HREC_EXP_SHIFT 21       /* window record: true exponent */

/* Huffman sub-table entry (u32), see above. */
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

/* Exponent blob (kind 5): BF16 weights whose exponent goes through rANS tiles under
 * a top-t table.  Rows padded to k_pad (a multiple of EC_RANS_ROW_ALIGN) with zero
 * weights; rANS positions as above (position 32 i + l of a tile is lane l's step i).
 * Table section: 2^prob_bits slot entries (bits 0..7 = the exponent itself for single
 * symbols, or the pair symbol 16 r0 + r1 of the exponents' ranks r0 (step 2m), r1
 * (step 2m + 1) in the ascending top-t table; bits 8..19 = slot - cum[s]; bits
 * 20..31 = freq[s] - 1), then 256 u32 holding, for pair symbol s, the two exponents
 * where a BF16 pair [w(2m+1) | w(2m)] keeps them (e0 << 7 | e1 << 23).  The section at
 * scales_off holds the sign / mantissa bytes: per tile EC_RAW_BYTES(steps) bytes in
 * the lane-transposed, pair-shuffled layout of the Huffman tiles (lane l's symbol i
 * at position 32 i + l).  Records as FP8 (u32 offsets per tile at esc_off_off, u32
 * records at esc_records_off), each = position in the tile | BF16 pattern << 16 of a
 * weight whose exponent is outside the table (coded as exponent 0, the table's first
 * entry).  fp8_table_size = the table size t, rans_tuple = 1 or 2; rANS tile records
 * (32 states, u16 words) last. */

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
    int32_t max_code_bytes;           /* Huffman: largest records + code area of any tile (bytes) */
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
    int64_t n_escapes;                /* FP8 and Huffman: correction records */
    int32_t huff_flags;               /* Huffman: EC_HUFF_WINDOW_REC */
    int32_t huff_sub_tables;          /* Huffman: hierarchical sub-tables after the pair table */
    int32_t huff_fill;                /* Huffman with window records: the exponent coded in place of a recorded one */
    int32_t max_code_area;            /* Huffman: largest code area of any tile (records excluded) */
    int32_t rans_values;              /* rANS 4-bit codes: EC_RANS_VALUES_INT4 (code + 8 in a symbol) or
                                       * EC_RANS_VALUES_FP4_E2M1 (the symbol is the E2M1 pattern) */
    uint8_t pad[256 - 4 * 4 - 8 * 10 - 4 * 8 - 8 * 3 - 4 * 5];
} ec_blob_header;

#endif /* EC_FORMAT_H_ */
