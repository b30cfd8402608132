/*
 * ec.h -- C ABI of the entropy-coded weight library (GB300, sm_103a).
 *
 * The library stores LLM weight matrices losslessly entropy-coded in GPU memory
 * and decodes them on the fly: either to dense BF16 (ec_decode) or fused into a
 * matrix-vector product y = W x (ec_gemv), so the dense weights never travel
 * through HBM.
 *
 * Two codecs:
 *  - Huffman over the BF16 exponent byte, sign and mantissa kept as one raw
 *    byte per weight.  Source: DFloat11, "70% Size, 100% Accuracy: Lossless LLM
 *    Compression for Efficient GPU Inference via Dynamic-Length Float", section
 *    "Dynamic-Length Float" (Fig. 3), decoding through hierarchical lookup
 *    tables (appendix, Fig. 13/14) with per-thread start offsets (section
 *    "two-phase kernel", Fig. 5, Algorithm 1).
 *  - Interleaved rANS in independent tiles for 4-bit codes with FP16 group
 *    scales.  Source: EntroPack (arXiv 2609.34185), section 3.6 and appendix
 *    C.3 (32 terminal states and a payload offset per tile, 32-bit states,
 *    16-bit payload words).
 * The fused decode + multiply-accumulate follows MINE ("Entropy-coded
 * Memory-efficient Inference for LLMs"), section 4 "Fused mvm" (Fig. 2).
 *
 * Conventions (all entry points):
 *  - Return EC_OK (0) or a negative EC_ERR_* code; no exception crosses the ABI.
 *  - Shapes are checked with overflow-safe 64-bit arithmetic before anything is
 *    allocated.
 *  - Device pointers are plain CUDA device addresses on the matrix's device;
 *    x and y must be 16-byte aligned.  The caller owns x, y, out and the stream.
 *  - Calls that take a stream are asynchronous on it.  Encoders synchronise
 *    their own upload before returning.
 *  - Corruption that only the GPU can see (payload bits) never faults or hangs
 *    a kernel: loops are bounded, reads are clamped to the matrix's buffer, and
 *    a device status word records EC_ERR_CORRUPT; ec_status() returns it.
 *
 * Environment (read once per process; both leave results unchanged):
 *  - EC_NO_PDL=1 launches every kernel without programmatic dependent launch
 *    (by default a kernel's prologue overlaps the end of the previous kernel in
 *    the stream, and it waits for that kernel before touching x, y or outputs).
 *  - EC_MMA_MIN_BATCH=n moves the batch from which the Huffman GEMV takes the
 *    tensor cores (default 6; above EC_MAX_BATCH: never).
 */
#ifndef EC_H_
#define EC_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#ifndef __DRIVER_TYPES_H__
typedef struct CUstream_st* cudaStream_t; /* same type as CUDA's cudaStream_t */
#endif

enum {
    EC_OK = 0,
    EC_ERR_INVALID_ARG = -1, /* null / misaligned pointer, bad parameter value */
    EC_ERR_SHAPE = -2,       /* negative or inconsistent dimensions */
    EC_ERR_OVERFLOW = -3,    /* a size computation would overflow */
    EC_ERR_UNSUPPORTED = -4, /* valid request the library does not implement (e.g. batch > 16) */
    EC_ERR_CORRUPT = -5,     /* the compressed data is inconsistent */
    EC_ERR_CUDA = -6,        /* a CUDA runtime call failed */
    EC_ERR_OOM = -7          /* host or device allocation failed */
};

#define EC_MAX_BATCH 64
#define EC_DEFAULT_MAX_CODE_LEN 12
#define EC_MAX_GROUP 8
#define EC_MAX_DECODE_BATCH 64

typedef struct ec_matrix ec_matrix; /* opaque: host descriptor + one device blob */

/* Huffman-exponent codec parameters (NULL = defaults).
 *  max_code_len  longest codeword, 1..24 (default EC_DEFAULT_MAX_CODE_LEN = 12);
 *                the code is textbook Huffman when it fits, otherwise the
 *                optimal length-limited code (package-merge).
 *  tile_steps    symbols per lane in one tile of 32 lanes: a multiple of 16 up
 *                to 256; 0 (the default) to choose by size: 128 (4096-weight
 *                tiles, 0.125 bit per weight of lane offsets) for matrices of at
 *                least 4 M padded weights, 64 from 2 M, else 32, so that a matrix
 *                has about 1024 tiles or more to spread over the SMs, then lowered
 *                in steps of 16 until 32 * tile_steps divides the padded row (for
 *                K = 14336: 112), so that no tile crosses a row; only such
 *                matrices take the tensor-core GEMV (ec_gemv), when the code
 *                areas of 31 rows of a tile column fit its staging pools.  Tiles
 *                of up to 256 steps carry fewer lane offsets (0.0625 bit per
 *                weight at 256), but the batch-1 GEMV runs fastest on 128.
 *  hierarchical  0 (default): the decoder reads two codewords per lookup of a
 *                12-bit window and never branches on the data.  Where a lane's two
 *                consecutive codewords overflow the window (about 0.6 % of pairs
 *                on LLM weights; also every codeword longer than 12 bits), the
 *                encoder codes the shortest-coded exponent instead and keeps the
 *                true one in a 32-bit correction record of the tile (MINE section
 *                4, "Escapes"), about 0.08 bit per weight.  When two of the
 *                shortest codewords exceed 12 bits (exponents nearly uniform) the
 *                encoder takes the hierarchical mode instead.
 *                1: no records; pairs that overflow the window and longer
 *                codewords are decoded through DFloat11's hierarchical tables
 *                (appendix, Fig. 14: 8-bit sub-tables behind the 12-bit first
 *                level), one data-dependent branch per pair. */
typedef struct {
    int32_t max_code_len;
    int32_t tile_steps;
    int32_t hierarchical;
    int32_t reserved;
} ec_huff_params;

/* rANS codec parameters (NULL = defaults).
 *  prob_bits         frequency precision b, 9..15 (default 12), or 0 to choose it per
 *                    matrix as MINE tunes its table size (section 4.2 "Launch"): b = 9..12
 *                    in increasing order, scored by the cross-entropy bound of the
 *                    stored size (payload n * H(P, Q_b) plus 2^b 4-byte table entries)
 *                    until a score exceeds the best so far by more than 1%; the best wins
 *  tile_syms         codes per independent tile, a multiple of 128 (default 4096)
 *  group             weights per FP16 scale along a row (only 128 is supported)
 *  codes_per_symbol  1 (default; 0 means 1): one 4-bit code per rANS symbol;
 *                    2: a symbol is the pair of a lane's consecutive codes (MINE's
 *                    k-tuple symbols), 256 symbols, half the decode steps, at
 *                    about 0.01 bit per code over single codes with b = 12
 *  values            what a 4-bit code means: EC_RANS_VALUES_INT4 (default, 0): a
 *                    signed integer, codes_host in [-8, 7] (int2 and int3 codes are
 *                    the subranges [-2, 1] and [-4, 3]); EC_RANS_VALUES_FP4_E2M1: an
 *                    FP4 E2M1 pattern (OCP Microscaling: sign, 2 exponent bits of bias
 *                    1, 1 mantissa bit), codes_host in [0, 15]; the weight is the
 *                    code's value times its group's FP16 scale (MINE, "Data Types") */
#define EC_RANS_VALUES_INT4 0
#define EC_RANS_VALUES_FP4_E2M1 1
typedef struct {
    int32_t prob_bits;
    int32_t tile_syms;
    int32_t group;
    int32_t codes_per_symbol;
    int32_t values;
} ec_rans_params;

/* E8 lattice codec parameters (NULL = defaults).
 *  prob_bits         frequency precision b of the 17 tables, 9..12 (default 11,
 *                    EntroPack's starting precision for rates up to 7 bits)
 *  tile_vectors      8-weight vectors per independent rANS tile, a multiple of 32
 *                    up to 1024 (default 1024: 8192 weights, so the 132 bytes of
 *                    terminal states and offset per tile stay near 3 % of a 4-bit
 *                    stream, within EntroPack's reported range); the bound keeps the
 *                    longest possible tile (12 bits for each of its 9 symbols a
 *                    vector) within the decoder's shared-memory buffers */
typedef struct {
    int32_t prob_bits;
    int32_t tile_vectors;
    int32_t reserved[2];
} ec_e8_params;

enum { EC_KIND_HUFFMAN_BF16 = 1, EC_KIND_RANS_INT4 = 2, EC_KIND_E8 = 3, EC_KIND_RANS_FP8 = 4, EC_KIND_RANS_EXP = 5 };

/* Parameters of the rANS codec for BF16 exponents (NULL = defaults).
 *  prob_bits   frequency precision b, 9..12 (default 12)
 *  tile_syms   weights per rANS tile, a multiple of 128 up to 4096 (default 4096)
 *  top_t       exponents kept in the decoding table, exponent 0 always among them:
 *              1..256 with single symbols, 1..16 with pairs; 0 (default) takes the
 *              smallest t with the least bound of the coded size, the cross-entropy
 *              of the symbol stream under the normalised table plus 32 bits per
 *              escape (MINE section 4.2, "Tuning t")
 *  single      0 (default): a symbol is the pair of exponents of a lane's two
 *              consecutive weights (MINE's "Pair" symbols; t^2 <= 2^prob_bits, and
 *              this format's 8-bit symbol field limits t to 16); 1: one exponent per
 *              symbol */
typedef struct {
    int32_t prob_bits;
    int32_t tile_syms;
    int32_t top_t;
    int32_t single;
} ec_exp_params;

/* FP8 codec parameters (NULL = defaults).
 *  prob_bits         frequency precision b, 9..12 (default 12)
 *  tile_syms         weights per rANS tile, a multiple of 128 up to 4096 (default 4096)
 *  top_t             codes kept in the decoding table, 1..256, code 0 always among
 *                    them (MINE section 4, "Escapes"); 0 (default) keeps every code
 *                    present.  A weight whose code is not kept is coded as 0 and
 *                    restored from a 32-bit correction record. */
typedef struct {
    int32_t prob_bits;
    int32_t tile_syms;
    int32_t top_t;
    int32_t reserved;
} ec_fp8_params;

/* Output dtypes of ec_decode_as. */
enum { EC_DTYPE_BF16 = 0, EC_DTYPE_FP8_E4M3 = 1, EC_DTYPE_INT8 = 2 };

/* Sizes and rates of one encoded matrix (ec_stats). */
typedef struct {
    int32_t kind;
    int32_t max_code_len;      /* longest codeword in use (Huffman) or prob_bits (rANS) */
    int64_t n_rows, k_cols;
    int64_t k_pad;             /* row length in the coded layout (zero padding at the row end) */
    int64_t n_tiles;
    int64_t payload_bits;      /* entropy-coded bits (exponent codewords or rANS words) */
    int64_t raw_bytes;         /* sign/mantissa bytes (Huffman) or 0 */
    int64_t aux_bytes;         /* per-tile offsets, lane starts, states, padding */
    int64_t table_bytes;       /* decode tables, group scales */
    int64_t device_bytes;      /* whole device blob */
    double bits_per_weight;    /* device_bytes * 8 / (n_rows * k_cols) */
    double entropy_bits;       /* H of the coded symbol (exponent byte or 4-bit code), Eq.(2) */
    double coded_bits_per_symbol; /* payload_bits / coded symbols */
    int64_t n_records;         /* 32-bit correction records (FP8 escapes, Huffman window records),
                                * counted in aux_bytes */
} ec_stats_t;

/* Encode a row-major BF16 matrix [n_rows, k_cols] (host memory, bit patterns) with
 * the Huffman-exponent codec and upload it to `device` (DFloat11, "Dynamic-Length
 * Float", Fig. 3: Huffman codes for the exponent byte, sign and mantissa stored as
 * they are; Eq. 2 bounds the size; length-limited codes as in its appendix).  The
 * stream is cut into tiles of 32 lanes with stored start offsets (the "stored by the
 * encoder" form of the per-thread positions of Algorithm 1's first phase).  Every one
 * of the 65536 BF16 patterns round-trips exactly.  On success *out owns a device blob; free it
 * with ec_free.  device < 0 keeps the blob in host memory (no CUDA call is made;
 * such a matrix can be serialised and inspected but not decoded on a GPU). */
int ec_encode_bf16(const uint16_t* w_host, int64_t n_rows, int64_t k_cols, const ec_huff_params* params,
                   int device, ec_matrix** out);

/* Encode 4-bit codes [n_rows, k_cols] (int8 host values: in [-8, 7], or FP4 E2M1
 * patterns in [0, 15] with params->values = EC_RANS_VALUES_FP4_E2M1) with FP16 scales
 * [n_rows, ceil(k_cols / group)] (host, bit patterns) as rANS tiles and upload them.
 * The represented weight is w = value(code) * scale (exact in FP32). */
int ec_encode_rans(const int8_t* codes_host, const uint16_t* scales_f16_host, int64_t n_rows, int64_t k_cols,
                   const ec_rans_params* params, int device, ec_matrix** out);

/* Encode E8 lattice points (EntroPack sections 3.2-3.7): row i of the matrix is
 * cut into blocks of 8 weights, each w = s * r_i * p with p in E8 = D8 u (D8 + 1/2)
 * (D8: integer vectors with an even sum).  q2_host [n_rows, k_cols] (host, int8,
 * k_cols % 8 == 0) holds q = 2 p; row_scales_host [n_rows] are the FP32 r_i and
 * `scale` the shared s.  Each point is coded as its coset c, seven coordinates
 * z_j = (q_j - c) / 2 in -16..15 and m = (z_8 - (z_1 + .. + z_7) mod 2) / 2 in -8..7,
 * with 17 frequency tables (c; each field under each coset) over independent rANS
 * tiles.  A decode (ec_decode / ec_decode_batch) writes bf16(fp32(q * fp32(s * r_i))
 * * 0.5).  Points outside that range or not in E8, a non-finite scale, or a row whose
 * fp32(s * r_i) is not finite: EC_ERR_INVALID_ARG.  ec_gemv and
 * ec_gemv_group on these matrices return EC_ERR_UNSUPPORTED (EntroPack decodes to a
 * dense matrix before its matrix products). */
int ec_encode_e8(const int8_t* q2_host, const float* row_scales_host, float scale, int64_t n_rows, int64_t k_cols,
                 const ec_e8_params* params, int device, ec_matrix** out);

/* Encode FP8 E4M3 weights: codes_host [n_rows, k_cols] (host, OCP E4M3 bytes; the NaN
 * pattern S.1111.111 is refused with EC_ERR_INVALID_ARG) with FP32 row scales
 * row_scales_host [n_rows] (finite), weight = fp32(value(code)) * r_i.  The codes kept
 * by the top-t table (params->top_t) go through interleaved rANS tiles (32 lanes,
 * 16-bit renormalisation, as ec_encode_rans); the others are coded as code 0 and
 * listed per tile as records (position in the tile | code << 16).  ec_gemv applies the
 * records inside the same kernel (batch 1..EC_MAX_BATCH, FP32 accumulation, y = r_i *
 * sum_j value * x); ec_decode writes bf16(fp32(value * r_i)).  Errors as ec_encode_rans. */
int ec_encode_fp8(const uint8_t* codes_host, const float* row_scales_host, int64_t n_rows, int64_t k_cols,
                  const ec_fp8_params* params, int device, ec_matrix** out);

/* Encode a row-major BF16 matrix [n_rows, k_cols] (host, bit patterns) with the
 * exponent going through rANS tiles under a top-t table and sign and mantissa kept
 * as one plain byte (MINE section 4: dtANS-LLM's BF16 handling; "Escapes": an
 * exponent outside the table is coded as exponent 0 and its weight listed in a
 * per-tile 32-bit record, position | BF16 pattern << 16; "Pair" symbols).  The
 * coding is lossless: every BF16 pattern round-trips.  ec_gemv / ec_gemv_group
 * (CUDA cores, batch 1..EC_MAX_BATCH, the records folded into each row's sum),
 * ec_decode, ec_decode_batch and ec_gemm accept the result.  Errors as
 * ec_encode_bf16; parameters out of range give EC_ERR_INVALID_ARG. */
int ec_encode_bf16_exp(const uint16_t* w_host, int64_t n_rows, int64_t k_cols, const ec_exp_params* params,
                       int device, ec_matrix** out);

/* Decode W to dense row-major BF16 [n_rows, k_cols] in device memory out_bf16
 * (DFloat11 Algorithm 1, second phase: table lookups, then sign | exponent |
 * mantissa reassembled and written at each symbol's output position; EntroPack
 * section 3.6 for the rANS tiles).
 * Huffman: the original bit patterns.  rANS: BF16 round-to-nearest-even of
 * code * scale.  FP8: of fp32(value * r_i), correction records applied.  E8: as
 * ec_decode_as with EC_DTYPE_BF16. */
int ec_decode(const ec_matrix* W, uint16_t* out_bf16, cudaStream_t stream);

/* Decode `count` matrices (1..EC_MAX_DECODE_BATCH) in one launch, the way
 * DFloat11 decompresses a whole transformer block at once (section
 * "Transformer-block-level decompression").  outs[m] is [n_rows(m), k_cols(m)]. */
int ec_decode_batch(const ec_matrix* const* Ws, uint16_t* const* outs, int count, cudaStream_t stream);

/* Decode W into device memory `out` [n_rows, k_cols] in `dtype` (EntroPack section
 * 3.7 and appendix B.1: the decoder writes floating-point or integer weights):
 *  EC_DTYPE_BF16      uint16 BF16 bit patterns, as ec_decode;
 *  EC_DTYPE_FP8_E4M3  uint8 OCP FP8 E4M3 codes of v = fp32(fp32(q) * fp32(s * r_i)) * 0.5,
 *                     nearest with ties to even, magnitudes beyond 448 saturating to 448;
 *  EC_DTYPE_INT8      int8 round-half-even of v, saturated to [-128, 127].
 * FP8 and INT8 are for E8 matrices (EC_ERR_UNSUPPORTED for the other kinds).  out must
 * be 16-byte aligned (EC_ERR_INVALID_ARG otherwise, or for an unknown dtype).  Async on
 * `stream`; corruption found on the device is reported by ec_status. */
int ec_decode_as(const ec_matrix* W, void* out, int dtype, cudaStream_t stream);

/* y[b, i] = sum_j W[i, j] * x[b, j] for b < batch (1..EC_MAX_BATCH), with the weights
 * decoded in registers / shared memory and FP32 accumulation (MINE section 4, "Fused
 * mvm": the decoded weight goes straight into the multiply-accumulate and never to
 * global memory).  Deviation from the proposed boundary: batches above 16 are
 * accepted, up to EC_MAX_BATCH.  x: BF16 [batch,
 * k_cols] device; y: FP32 [batch, n_rows] device, overwritten.
 * Huffman matrices run on the CUDA cores (one FMA per weight and batch row, in
 * passes of up to 16 rows), or, from batch 6 (EC_MMA_MIN_BATCH overrides) when
 * every tile lies inside a row (the automatic tile size ensures it) and k_cols % 8
 * == 0, on the tensor cores (tcgen05, BF16 products, FP32 accumulators; passes of
 * up to 32 rows).  ec_gemv_path tells which.  rANS and FP8 matrices run on the CUDA
 * cores; E8 matrices return EC_ERR_UNSUPPORTED (decode them instead). */
int ec_gemv(const ec_matrix* W, const uint16_t* x_bf16, float* y, int batch, cudaStream_t stream);

enum { EC_PATH_CUDA_CORES = 1, EC_PATH_TENSOR_CORES = 2 };

/* The kernel family ec_gemv_group(Ws, count, ..., batch, ...) would use (host only;
 * no device access): EC_PATH_*, or a negative EC_ERR_* for arguments it rejects
 * before launching (null or mixed matrices, batch out of range). */
int ec_gemv_path(const ec_matrix* const* Ws, int count, int batch);

/* Several GEMVs over the same input x in one launch (MINE section 4.2 "Launch":
 * q/k/v, gate/up).  All matrices must have the same kind and k_cols; count <=
 * EC_MAX_GROUP; ys[m] is [batch, n_rows(m)]. */
int ec_gemv_group(const ec_matrix* const* Ws, int count, const uint16_t* x_bf16, float* const* ys, int batch,
                  cudaStream_t stream);

/* Allocation-free GEMV.  Same result contract as ec_gemv (Huffman-coded matrices,
 * batch 1..EC_MAX_BATCH, y overwritten), for callers that must not allocate device
 * memory while serving: a cudaMalloc can stall the whole device and can fail at an
 * arbitrary point, and some processes hand all device memory to one allocator (for
 * example a framework's caching allocator) or reserve a fixed budget up front.
 * This call allocates nothing, on the device or the host.  Its working memory is a
 * fixed 4 MiB array built into the library (every GPU that loads the library keeps
 * it until the process exits): a status word plus one partial sum per (batch row,
 * output row, tile covering that row); the tiles' partial sums are added in tile
 * order by a second small kernel, so repeated calls give identical y.
 * Limits: batch * n_rows * (ceil(k_pad / tile) + 1) partial sums must fit in that
 * array (about 1M floats), otherwise EC_ERR_UNSUPPORTED; rANS, FP8 and E8 matrices
 * also return EC_ERR_UNSUPPORTED.  The first call on a device looks up the array's device
 * address (cudaGetSymbolAddress) and the device's limits once; make that first call
 * before any stream capture.  All calls share the one array: calls whose work
 * overlaps on the GPU (other streams, other threads) race and corrupt each other's
 * partial sums, so serialise them.  Corruption found in the payload is recorded in
 * the array's status word, which stays set until ec_status() reads and clears it
 * (together with the regular one).  The pages have no counterpart to this entry
 * point. */
int ec_gemv_static(const ec_matrix* W, const uint16_t* x_bf16, float* y, int batch, cudaStream_t stream);

/* Uncompressed comparator: y = W x for a dense BF16 W [n_rows, k_cols] in device
 * memory, FP32 accumulation, same x / y conventions as ec_gemv. */
int ec_bf16_gemv(const uint16_t* w_bf16, int64_t n_rows, int64_t k_cols, const uint16_t* x_bf16, float* y,
                 int batch, cudaStream_t stream);

/* Prefill / batched products: y[b, i] = sum_j W[i, j] * x[b, j] for any batch >= 1
 * (MINE section 4: at batch > 1 the layer is materialised, then multiplied by a
 * GEMM; DFloat11 "Transformer-block-level decompression").  Huffman matrices are
 * decoded in chunks of rows (about 48 MB of BF16, so a chunk stays in the 129 MB
 * L2 between its decode and its use) into `work`, and each chunk is multiplied on
 * the tensor cores (tcgen05, BF16 products, FP32 accumulators in tensor memory)
 * before the next chunk is decoded; rANS, FP8 and E8 matrices are decoded whole
 * (k_cols % 8 == 0, else EC_ERR_UNSUPPORTED).  When K is split across CTAs the
 * partial sums go to `work` and are added in a fixed order, so repeated calls
 * give identical y.  x: BF16 [batch, k_cols], y: FP32 [batch, n_rows] (device,
 * 16-byte aligned, y overwritten).  work: device memory owned by the caller,
 * 16-byte aligned, work_bytes at least ec_gemm_work_bytes() for the full chunk
 * size; a smaller buffer makes the chunks smaller (EC_ERR_INVALID_ARG when not even
 * one chunk of the minimum height fits).  Asynchronous on `stream`; allocates
 * nothing; corruption is reported by ec_status. */
int ec_gemm(const ec_matrix* W, const uint16_t* x_bf16, float* y, int batch, void* work, size_t work_bytes,
            cudaStream_t stream);

/* Work bytes ec_gemm(W, ..., batch, ...) uses with full-size chunks on the current
 * device (host only). */
int ec_gemm_work_bytes(const ec_matrix* W, int batch, size_t* bytes);

/* ec_gemm over `count` matrices (1..EC_MAX_DECODE_BATCH), ys[m] = xs[m] W_m^T at the
 * same batch (x and y per matrix: a transformer block's matrices take different
 * inputs).  Huffman matrices with k_cols % 8 == 0 whose decoded rows fit in `work`
 * together (beside the partial sums) are decoded in one launch, as ec_decode_batch
 * decodes a block (DFloat11, "Transformer-block-level decompression"), then
 * multiplied one after the other; any other matrix goes through ec_gemm on its own,
 * in row chunks.  ec_gemm_group_work_bytes gives the size that decodes every
 * packable matrix in one launch; less work memory makes more launches.  Results as
 * ec_gemm. */
int ec_gemm_group(const ec_matrix* const* Ws, int count, const uint16_t* const* xs_bf16, float* const* ys,
                  int batch, void* work, size_t work_bytes, cudaStream_t stream);
int ec_gemm_group_work_bytes(const ec_matrix* const* Ws, int count, int batch, size_t* bytes);

/* Uncompressed comparator for ec_gemm: y = W x for a dense BF16 W [n_rows, k_cols]
 * (k_cols % 8 == 0, else EC_ERR_UNSUPPORTED) through the same tensor-core GEMM.
 * work (may be NULL) holds partial sums when K is split: with less than
 * splits * batch * n_rows floats the split is reduced. */
int ec_bf16_gemm(const uint16_t* w_bf16, int64_t n_rows, int64_t k_cols, const uint16_t* x_bf16, float* y,
                 int batch, void* work, size_t work_bytes, cudaStream_t stream);

/* Sizes and rates (host only): the stored bytes by section, bits per weight, and
 * the exponent entropy H of DFloat11 Eq. 2 (or of the 4-bit code for rANS), so
 * that the coded rate can be checked against the entropy bound. */
int ec_stats(const ec_matrix* W, ec_stats_t* out);

/* Code length of each exponent value (Huffman matrices; 0 = absent). */
int ec_code_lengths(const ec_matrix* W, uint8_t lengths[256]);

/* Synchronise `stream`, then return and clear the device status words of the
 * current device (the regular one and that of ec_gemv_static): EC_OK, or
 * EC_ERR_CORRUPT if a kernel met inconsistent data (a lane whose codewords do not
 * end at the next lane's stored start, a tile record out of range, an rANS tile
 * whose final states differ from the initial value: the consistency checks that the
 * per-tile offsets of DFloat11 Algorithm 1 and the terminal states of EntroPack
 * section 3.6 make possible). */
int ec_status(cudaStream_t stream);

/* Serialise W into host memory: a fixed metadata block followed by the device blob
 * (copied back from the GPU).  With dst == NULL only *size_out is set.  Fails with
 * EC_ERR_INVALID_ARG if capacity < *size_out. */
int ec_serialize(const ec_matrix* W, void* dst, int64_t capacity, int64_t* size_out);

/* Rebuild a matrix from ec_serialize output.  The bytes are untrusted: the
 * metadata, every section offset, every tile offset and every decode-table entry
 * are validated before anything is allocated or uploaded (EC_ERR_CORRUPT on any
 * inconsistency).  device < 0 keeps the blob in host memory (inspection only;
 * ec_decode / ec_gemv reject such a matrix). */
int ec_deserialize(const void* src, int64_t size, int device, ec_matrix** out);

/* Free a matrix (host descriptor and device blob). NULL is ignored. */
void ec_free(ec_matrix* W);

/* Human-readable text for an EC_* code. */
const char* ec_strerror(int code);

#ifdef __cplusplus
}
#endif
#endif /* EC_H_ */
