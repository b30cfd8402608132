/*
 * oracle.c -- plain, slow CPU reference for the entropy-coded weight path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library (lossless_entropy_coded_gb300)
 * includes, links or calls this file; only tests/, the smoke check and the
 * benchmark's CPU-baseline leg load it.  It shares no code, header, table or
 * constant generator with the CUDA path.
 *
 * What it follows (sources are the pages' titles and sections):
 *  - DFloat11, "70% Size, 100% Accuracy: Lossless LLM Compression for Efficient
 *    GPU Inference via Dynamic-Length Float": Eq.(1) BF16 field split; Eq.(2)
 *    Shannon entropy; the Huffman exponent coding with sign and mantissa kept as
 *    a raw byte (section "Dynamic-Length Float", Fig. 3); the flat LUT plus
 *    CodeLengths (appendix "two lookup tables", Fig. 13); hierarchical compact
 *    LUTs of b bits each (appendix, Fig. 14); per-thread byte chunks with Gaps
 *    and BlockOutputPos (section "two-phase kernel", Fig. 5); the two-phase
 *    decompression of Algorithm 1.
 *  - EntroPack (arXiv 2609.34185), section 3.6 and appendix C.3: independent
 *    rANS tiles, 32 terminal states plus a 32-bit payload offset per tile,
 *    32-bit states, 16-bit payload words, at most one word per symbol.
 *  - rANS itself: Duda, "Asymmetric numeral systems" (2013), cited by MINE
 *    section 3.
 *
 * Readings of points the pages leave open are marked "reading:" below.
 * Floating point: every sum is an FP64 sum in index order.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ===========================================================================
 * Storage-type helpers (IEEE definitions written out).
 * ========================================================================= */

/* BF16 bit pattern -> value: the top 16 bits of an FP32 (DFloat11 Eq. (1)). */
double orc_bf16_to_f64(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* FP16 bit pattern -> FP32 value, from the binary16 definition. */
float orc_f16_to_f32(uint16_t h) {
    const int s = (h >> 15) & 1, e = (h >> 10) & 0x1F, m = h & 0x3FF;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24); /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp(1024.0 + m, e - 25); /* (1 + m/1024) * 2^(e-15) */
    return (float)(s ? -v : v);
}

/* FP32 -> BF16 with round-to-nearest, ties to even (NaN stays NaN). */
uint16_t orc_f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if (isnan(f)) return (uint16_t)((u >> 16) | 0x40);
    const uint32_t lower = u & 0xFFFFu, upper = u >> 16;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) return (uint16_t)(upper + 1u);
    return (uint16_t)upper;
}

/* FP32 -> FP8 E4M3 of the OCP 8-bit floating-point format: 1 sign bit, 4 exponent
 * bits with bias 7, 3 mantissa bits; exponent field 0 holds the subnormals m/8 * 2^-6;
 * S.1111.111 is NaN, so the largest finite magnitude is 1.75 * 2^8 = 448, and there are
 * no infinities.  Rounding: the nearest finite code, ties to the even code ("satfinite":
 * magnitudes beyond 448, infinities included, give 448).  The sign bit is the input's
 * (so -0 and negative values rounding to zero give 0x80); NaN gives 0x7F | sign. */
static double e4m3_value(int code) { /* magnitude of code 0..126 */
    const int e = code >> 3, m = code & 7;
    return e == 0 ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, e - 7);
}

uint8_t orc_f32_to_e4m3_satfinite(float f) {
    const uint8_t sign = signbit(f) ? 0x80u : 0u;
    if (isnan(f)) return (uint8_t)(sign | 0x7Fu);
    const double a = fabs((double)f);
    if (a >= 448.0) return (uint8_t)(sign | 0x7Eu); /* the largest finite value is the nearest */
    int best = 0;
    double best_d = a;
    for (int c = 1; c <= 126; ++c) {
        const double d = fabs(e4m3_value(c) - a);
        if (d < best_d || (d == best_d && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            best_d = d;
        }
    }
    return (uint8_t)(sign | (uint8_t)best);
}

/* FP32 -> INT8: the nearest integer, ties to even, saturated to [-128, 127] (NaN: 0). */
int8_t orc_f32_to_s8_rne_sat(float f) {
    if (isnan(f)) return 0;
    if (f >= 127.0f) return 127;
    if (f <= -128.0f) return -128;
    const double a = (double)f, r = floor(a), d = a - r;
    double n = r;
    if (d > 0.5 || (d == 0.5 && fmod(r, 2.0) != 0.0)) n = r + 1.0;
    return (int8_t)n;
}

/* ===========================================================================
 * Entropy (DFloat11 Eq. (2); MINE section 3: H(P) lower-bounds the size).
 * ========================================================================= */
double orc_entropy(const uint64_t* counts, int n_symbols) {
    double total = 0.0, h = 0.0;
    for (int s = 0; s < n_symbols; ++s) total += (double)counts[s];
    if (total <= 0.0) return 0.0;
    for (int s = 0; s < n_symbols; ++s) {
        if (!counts[s]) continue;
        const double p = (double)counts[s] / total;
        h -= p * log2(p);
    }
    return h;
}

/* Cross-entropy (bits/symbol) of empirical counts under model q_s = f_s / 2^prob_bits
 * (MINE section 4.2 "Compressed Size Prediction"). Returns INFINITY if a present
 * symbol has f_s = 0. */
double orc_cross_entropy(const uint64_t* counts, const uint32_t* freqs, int n_symbols, int prob_bits) {
    double total = 0.0, h = 0.0;
    for (int s = 0; s < n_symbols; ++s) total += (double)counts[s];
    if (total <= 0.0) return 0.0;
    for (int s = 0; s < n_symbols; ++s) {
        if (!counts[s]) continue;
        if (!freqs[s]) return INFINITY;
        h -= (double)counts[s] / total * (log2((double)freqs[s]) - prob_bits);
    }
    return h;
}

/* ===========================================================================
 * Huffman code lengths.
 * ========================================================================= */

/* Textbook Huffman (DFloat11 section "entropy coding": repeatedly merge the two
 * least frequent nodes).  reading: ties are broken by (weight, smallest symbol in
 * the subtree).  One present symbol gets length 1.  Returns the number of
 * present symbols; lengths of absent symbols are 0. */
int orc_huffman_textbook(const uint64_t counts[256], uint8_t lengths[256]) {
    uint64_t w[511];
    int minsym[511], parent[511], alive[511];
    int n = 0, leaf_of[256];
    memset(lengths, 0, 256);
    for (int s = 0; s < 256; ++s) {
        leaf_of[s] = -1;
        if (!counts[s]) continue;
        w[n] = counts[s];
        minsym[n] = s;
        parent[n] = -1;
        alive[n] = 1;
        leaf_of[s] = n++;
    }
    if (n == 0) return 0;
    if (n == 1) {
        for (int s = 0; s < 256; ++s)
            if (leaf_of[s] >= 0) lengths[s] = 1;
        return 1;
    }
    int total = n;
    for (int merges = 0; merges < n - 1; ++merges) {
        int a = -1, b = -1;
        for (int i = 0; i < total; ++i) {
            if (!alive[i]) continue;
            if (a < 0 || w[i] < w[a] || (w[i] == w[a] && minsym[i] < minsym[a])) {
                b = a;
                a = i;
            } else if (b < 0 || w[i] < w[b] || (w[i] == w[b] && minsym[i] < minsym[b])) {
                b = i;
            }
        }
        w[total] = w[a] + w[b];
        minsym[total] = minsym[a] < minsym[b] ? minsym[a] : minsym[b];
        parent[total] = -1;
        alive[total] = 1;
        alive[a] = alive[b] = 0;
        parent[a] = parent[b] = total;
        ++total;
    }
    for (int s = 0; s < 256; ++s) {
        if (leaf_of[s] < 0) continue;
        int d = 0;
        for (int v = leaf_of[s]; parent[v] >= 0; v = parent[v]) ++d;
        lengths[s] = (uint8_t)d;
    }
    return n;
}

/* Package-merge (Larmore & Hirschberg 1990), the optimal length-limited prefix
 * code, in its "coin collector" form.  Items are leaves (one per present symbol,
 * sorted by (weight, symbol)) and packages (adjacent pairs of the previous list).
 * reading: on equal weight a leaf precedes a package when merging.
 * The list for denomination 2^-1 keeps its first 2(n-1) items; a symbol's length
 * is the number of times its leaf occurs inside them.  Returns n, or -1 if
 * 2^max_len < n. */
typedef struct {
    uint64_t w;
    int leaf;      /* symbol, or -1 for a package */
    int child[2];  /* indices into the previous level's list */
} pm_item;

static void pm_count(pm_item* const* lists, int level, int idx, int* cnt) {
    const pm_item* it = &lists[level][idx];
    if (it->leaf >= 0) {
        cnt[it->leaf]++;
        return;
    }
    pm_count(lists, level - 1, it->child[0], cnt);
    pm_count(lists, level - 1, it->child[1], cnt);
}

int orc_package_merge(const uint64_t counts[256], int max_len, uint8_t lengths[256]) {
    int syms[256], n = 0;
    memset(lengths, 0, 256);
    for (int s = 0; s < 256; ++s)
        if (counts[s]) syms[n++] = s;
    if (n == 0) return 0;
    if (n == 1) {
        lengths[syms[0]] = 1;
        return 1;
    }
    if (max_len < 1 || max_len > 30 || (1LL << max_len) < n) return -1;
    /* leaves sorted by (weight, symbol): insertion sort */
    for (int i = 1; i < n; ++i) {
        int s = syms[i], j = i - 1;
        while (j >= 0 && (counts[syms[j]] > counts[s] || (counts[syms[j]] == counts[s] && syms[j] > s))) {
            syms[j + 1] = syms[j];
            --j;
        }
        syms[j + 1] = s;
    }
    /* lists[0] is denomination 2^-max_len (leaves only); lists[d] is 2^-(max_len-d). */
    pm_item** lists = (pm_item**)calloc((size_t)max_len, sizeof(pm_item*));
    int* sizes = (int*)calloc((size_t)max_len, sizeof(int));
    for (int d = 0; d < max_len; ++d) lists[d] = (pm_item*)malloc(sizeof(pm_item) * (size_t)(2 * n));
    for (int i = 0; i < n; ++i) {
        lists[0][i].w = counts[syms[i]];
        lists[0][i].leaf = syms[i];
    }
    sizes[0] = n;
    for (int d = 1; d < max_len; ++d) {
        const pm_item* prev = lists[d - 1];
        const int np = sizes[d - 1] / 2; /* packages: pairs (0,1), (2,3), ... */
        int li = 0, pi = 0, k = 0;
        while (li < n || pi < np) {
            const uint64_t pw = pi < np ? prev[2 * pi].w + prev[2 * pi + 1].w : 0;
            if (li < n && (pi >= np || counts[syms[li]] <= pw)) {
                lists[d][k].w = counts[syms[li]];
                lists[d][k].leaf = syms[li];
                ++li;
            } else {
                lists[d][k].w = pw;
                lists[d][k].leaf = -1;
                lists[d][k].child[0] = 2 * pi;
                lists[d][k].child[1] = 2 * pi + 1;
                ++pi;
            }
            ++k;
        }
        sizes[d] = k;
    }
    int cnt[256] = {0};
    for (int i = 0; i < 2 * (n - 1); ++i) pm_count(lists, max_len - 1, i, cnt);
    for (int s = 0; s < 256; ++s) lengths[s] = (uint8_t)cnt[s];
    for (int d = 0; d < max_len; ++d) free(lists[d]);
    free(lists);
    free(sizes);
    return n;
}

/* Lengths used by the codec: textbook Huffman if its longest code fits max_len,
 * else package-merge (reading: DFloat11 leaves the limit open; 24 is the
 * workload's stated maximum). */
int orc_code_lengths(const uint64_t counts[256], int max_len, uint8_t lengths[256]) {
    int n = orc_huffman_textbook(counts, lengths);
    int longest = 0;
    for (int s = 0; s < 256; ++s)
        if (lengths[s] > longest) longest = lengths[s];
    if (longest <= max_len) return n;
    return orc_package_merge(counts, max_len, lengths);
}

/* Canonical codewords: symbols sorted by (length, symbol) get consecutive
 * values, shifted left whenever the length grows.  This reproduces DFloat11
 * Fig. 13 (A=0, B=100, C=101, D=110, E=1110, F=1111). */
void orc_canonical_codes(const uint8_t lengths[256], uint32_t codes[256]) {
    uint32_t code = 0;
    int prev_len = 0, first = 1;
    memset(codes, 0, 256 * sizeof(uint32_t));
    for (int l = 1; l <= 32; ++l) {
        for (int s = 0; s < 256; ++s) {
            if (lengths[s] != l) continue;
            if (first) {
                code = 0;
                first = 0;
            } else {
                code = (code + 1) << (l - prev_len);
            }
            prev_len = l;
            codes[s] = code;
        }
    }
}

/* ===========================================================================
 * Lookup tables.
 * ========================================================================= */

/* Flat LUT of 2^L entries (DFloat11 appendix, Fig. 13): entry i holds the symbol
 * whose codeword is a prefix of the L-bit string i; -1 if none. */
int orc_flat_lut(const uint8_t lengths[256], const uint32_t codes[256], int L, int16_t* lut) {
    if (L < 1 || L > 24) return -1;
    for (int64_t i = 0; i < (1 << L); ++i) lut[i] = -1;
    for (int s = 0; s < 256; ++s) {
        const int l = lengths[s];
        if (!l) continue;
        if (l > L) return -1;
        const uint32_t lo = codes[s] << (L - l), hi = (codes[s] + 1) << (L - l);
        for (uint32_t i = lo; i < hi; ++i) lut[i] = (int16_t)s;
    }
    return 0;
}

/* Hierarchical LUTs, b bits per table (DFloat11 appendix "decomposing the LUT",
 * Fig. 4 and Fig. 14).  Table t has 2^b entries.  reading: an entry is a
 * 16-bit value -- 0..255 is a decoded exponent, 256+j points at table j, -1 is
 * unused -- so all 256 exponent values stay legal (the pages reserve 240..255 as
 * pointers, which cannot represent exponents 240..255).  Tables are numbered in
 * breadth-first order of their prefixes, children in index order.
 * Returns the number of tables, or -1 if more than max_tables are needed. */
int orc_hier_luts(const uint8_t lengths[256], const uint32_t codes[256], int b, int16_t* luts,
                  int max_tables) {
    if (b < 1 || b > 12) return -1;
    uint32_t prefix[4096];
    int depth[4096];
    int n_tables = 1, head = 0;
    prefix[0] = 0;
    depth[0] = 0;
    const int size = 1 << b;
    while (head < n_tables) {
        const int t = head++;
        const int d = depth[t];
        for (int v = 0; v < size; ++v) {
            /* bit string P.v of length d + b, compared with every codeword */
            const uint64_t pv = ((uint64_t)prefix[t] << b) | (uint64_t)v;
            const int dl = d + b;
            int16_t entry = -1;
            int needs_child = 0;
            for (int s = 0; s < 256; ++s) {
                const int l = lengths[s];
                if (!l) continue;
                if (l <= dl) {
                    if ((pv >> (dl - l)) == codes[s] && l > d) {
                        entry = (int16_t)s;
                        break;
                    }
                } else if (((uint64_t)codes[s] >> (l - dl)) == pv) {
                    needs_child = 1;
                }
            }
            if (entry < 0 && needs_child) {
                if (n_tables >= max_tables || n_tables >= 4096) return -1;
                prefix[n_tables] = (uint32_t)pv;
                depth[n_tables] = dl;
                entry = (int16_t)(256 + n_tables);
                ++n_tables;
            }
            luts[(size_t)t * size + v] = entry;
        }
    }
    return n_tables;
}

/* ===========================================================================
 * DFloat11 format: EncodedExponent, PackedSignMantissa, Gaps, BlockOutputPos.
 * ========================================================================= */
typedef struct {
    int64_t n;              /* number of weights */
    int n_bytes;            /* bytes per thread chunk (the pages' n) */
    int threads;            /* threads per block (the pages' T) */
    int64_t n_chunks, n_blocks;
    int64_t stream_bytes;   /* EncodedExponent length incl. padding */
    uint8_t* stream;        /* EncodedExponent, MSB-first */
    uint8_t* sm;            /* PackedSignMantissa: (sign << 7) | mantissa */
    uint16_t* gaps;         /* one per chunk, bit offset of its first codeword */
    uint64_t* block_pos64;  /* BlockOutputPos, n_blocks + 1 entries */
    uint8_t lengths[256];
    uint32_t codes[256];
    uint64_t counts[256];
    int16_t* luts;          /* hierarchical, b = 8 */
    int n_luts;
    int64_t payload_bits;   /* sum of codeword lengths */
} orc_df11;

void orc_df11_free(orc_df11* d) {
    if (!d) return;
    free(d->stream);
    free(d->sm);
    free(d->gaps);
    free(d->block_pos64);
    free(d->luts);
    free(d);
}

/* Encoder (DFloat11 section "Dynamic-Length Float" and Fig. 3/5).
 * Step 1: split w into the exponent byte e = (w >> 7) & 0xFF and the raw byte
 *         sm = ((w >> 8) & 0x80) | (w & 0x7F); count e over the whole matrix.
 * Step 2: code lengths (max_len), canonical codewords.
 * Step 3: concatenate codewords MSB-first into EncodedExponent.
 * Step 4: cut the stream into chunks of n_bytes; gap = offset of the first
 *         codeword starting in the chunk; BlockOutputPos[b] = index of the first
 *         element whose codeword starts in block b, BlockOutputPos[B] = n.
 * reading: the stream is padded with zero bytes to whole blocks plus 4 bytes, so
 * a 4-byte read at any chunk offset stays inside it. */
orc_df11* orc_df11_encode(const uint16_t* w, int64_t n, int max_len, int n_bytes, int threads) {
    if (n < 0 || n_bytes < 1 || threads < 1 || max_len < 1 || max_len > 24) return NULL;
    orc_df11* d = (orc_df11*)calloc(1, sizeof(orc_df11));
    d->n = n;
    d->n_bytes = n_bytes;
    d->threads = threads;
    for (int64_t p = 0; p < n; ++p) d->counts[(w[p] >> 7) & 0xFF]++;
    if (orc_code_lengths(d->counts, max_len, d->lengths) < 0) {
        orc_df11_free(d);
        return NULL;
    }
    orc_canonical_codes(d->lengths, d->codes);
    d->luts = (int16_t*)malloc(sizeof(int16_t) * 256 * 4096);
    d->n_luts = orc_hier_luts(d->lengths, d->codes, 8, d->luts, 4096);

    int64_t bits = 0;
    for (int64_t p = 0; p < n; ++p) bits += d->lengths[(w[p] >> 7) & 0xFF];
    d->payload_bits = bits;
    const int64_t block_bytes = (int64_t)n_bytes * threads;
    int64_t nbytes = (bits + 7) / 8;
    d->n_blocks = (nbytes + block_bytes - 1) / block_bytes;
    if (d->n_blocks == 0) d->n_blocks = 1;
    d->n_chunks = d->n_blocks * threads;
    d->stream_bytes = d->n_blocks * block_bytes + 4;
    d->stream = (uint8_t*)calloc((size_t)d->stream_bytes, 1);
    d->sm = (uint8_t*)malloc((size_t)(n > 0 ? n : 1));
    d->gaps = (uint16_t*)calloc((size_t)d->n_chunks, sizeof(uint16_t));
    d->block_pos64 = (uint64_t*)malloc(sizeof(uint64_t) * (size_t)(d->n_blocks + 1));
    for (int64_t b = 0; b <= d->n_blocks; ++b) d->block_pos64[b] = (uint64_t)n;

    /* Codewords MSB-first.  Elements are visited in increasing start bit, so the
     * first element starting at or after chunk c's first bit is the current one
     * for every chunk c not yet assigned whose first bit is <= its start. */
    const int64_t chunk_bits = 8 * (int64_t)n_bytes;
    int64_t bitpos = 0, next_chunk = 0;
    for (int64_t p = 0; p < n; ++p) {
        const int e = (w[p] >> 7) & 0xFF;
        d->sm[p] = (uint8_t)(((w[p] >> 8) & 0x80) | (w[p] & 0x7F));
        while (next_chunk < d->n_chunks && next_chunk * chunk_bits <= bitpos) {
            const int64_t off = bitpos - next_chunk * chunk_bits;
            /* reading: a chunk in which no codeword starts gets gap = 8n (decodes nothing) */
            d->gaps[next_chunk] = (uint16_t)(off < chunk_bits ? off : chunk_bits);
            if (next_chunk % threads == 0) d->block_pos64[next_chunk / threads] = (uint64_t)p;
            ++next_chunk;
        }
        const int l = d->lengths[e];
        const uint32_t c = d->codes[e];
        for (int k = l - 1; k >= 0; --k) {
            if ((c >> k) & 1u) d->stream[bitpos >> 3] |= (uint8_t)(0x80u >> (bitpos & 7));
            ++bitpos;
        }
    }
    /* Chunks after the last codeword start hold only padding: gap 0, and their
     * blocks start at n (already set); whatever they decode is dropped. */
    for (; next_chunk < d->n_chunks; ++next_chunk) d->gaps[next_chunk] = 0;
    return d;
}

/* Read the 32-bit MSB-first window starting at absolute bit `bit`. */
static uint32_t window32(const uint8_t* s, int64_t bit) {
    const int64_t byte = bit >> 3;
    const int sh = (int)(bit & 7);
    uint64_t v = 0;
    for (int i = 0; i < 5; ++i) v = (v << 8) | s[byte + i];
    return (uint32_t)(v >> (8 - sh));
}

/* Decoder: Algorithm 1 of DFloat11 ("DF11ToBF16"), both phases.
 * For block b and thread t: BitOffset starts at Gaps[bT+t]; while BitOffset < 8n,
 * read the 4 bytes of the window at BitOffset, look up LUT_1[Byte_1] and follow
 * pointers through Byte_2.. while the entry is a pointer, then advance by
 * CodeLengths[Exponent].  Phase 1 counts, an exclusive prefix sum over the
 * block's threads gives ThreadOutputPos, phase 2 decodes again and writes
 * (Sign << 8) | (Exponent << 7) | Mantissa into the block's write buffer, which is
 * copied to Outputs[BlockOutputPos[b] .. BlockOutputPos[b+1]).
 * reading: elements whose index reaches BlockOutputPos[b+1] are dropped (they
 * are padding bits of the last block).  Returns 0, or -1 on a bad table walk. */
int orc_df11_decode(const orc_df11* d, uint16_t* out) {
    if (d->n == 0) return 0; /* no elements, no code */
    const int T = d->threads, n = d->n_bytes;
    int64_t* num = (int64_t*)malloc(sizeof(int64_t) * (size_t)T);
    int64_t* pos = (int64_t*)malloc(sizeof(int64_t) * (size_t)T);
    uint16_t* wbuf = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(8 * n * T + 1));
    int rc = 0;
    for (int64_t b = 0; b < d->n_blocks && rc == 0; ++b) {
        const int64_t b_lo = (int64_t)d->block_pos64[b], b_hi = (int64_t)d->block_pos64[b + 1];
        for (int phase = 1; phase <= 2 && rc == 0; ++phase) {
            for (int t = 0; t < T && rc == 0; ++t) {
                const int64_t chunk = b * T + t;
                const int64_t base = chunk * 8 * (int64_t)n;
                int64_t off = d->gaps[chunk];
                if (phase == 1) num[t] = 0;
                while (off < 8 * (int64_t)n) {
                    const uint32_t win = window32(d->stream, base + off);
                    int i = 0;
                    int v = d->luts[(win >> 24) & 0xFF];
                    while (v >= 256) {
                        ++i;
                        if (i > 3) {
                            rc = -1;
                            break;
                        }
                        v = d->luts[(size_t)(v - 256) * 256 + ((win >> (24 - 8 * i)) & 0xFF)];
                    }
                    if (rc || v < 0) {
                        rc = -1;
                        break;
                    }
                    if (phase == 1) {
                        num[t]++;
                    } else {
                        if (pos[t] < b_hi) {
                            const uint8_t smb = d->sm[pos[t]];
                            wbuf[pos[t] - b_lo] =
                                (uint16_t)(((smb & 0x80u) << 8) | ((uint32_t)v << 7) | (smb & 0x7Fu));
                        }
                        pos[t]++;
                    }
                    off += d->lengths[v];
                }
            }
            if (phase == 1) { /* exclusive prefix sum over the block's threads */
                int64_t acc = b_lo;
                for (int t = 0; t < T; ++t) {
                    pos[t] = acc;
                    acc += num[t];
                }
            }
        }
        for (int64_t p = b_lo; p < b_hi && rc == 0; ++p) out[p] = wbuf[p - b_lo];
    }
    free(num);
    free(pos);
    free(wbuf);
    return rc;
}

/* Accessors for tests. */
int64_t orc_df11_info(const orc_df11* d, int64_t* out /* 8 */) {
    out[0] = d->n;
    out[1] = d->n_bytes;
    out[2] = d->threads;
    out[3] = d->n_chunks;
    out[4] = d->n_blocks;
    out[5] = d->stream_bytes;
    out[6] = d->payload_bits;
    out[7] = d->n_luts;
    return 0;
}
const uint8_t* orc_df11_lengths(const orc_df11* d) { return d->lengths; }
const uint32_t* orc_df11_codes(const orc_df11* d) { return d->codes; }
const uint64_t* orc_df11_counts(const orc_df11* d) { return d->counts; }
const uint8_t* orc_df11_stream(const orc_df11* d) { return d->stream; }
const uint16_t* orc_df11_gaps(const orc_df11* d) { return d->gaps; }
const uint64_t* orc_df11_block_pos(const orc_df11* d) { return d->block_pos64; }
const int16_t* orc_df11_luts(const orc_df11* d) { return d->luts; }
uint8_t* orc_df11_sm_mut(orc_df11* d) { return d->sm; }
uint8_t* orc_df11_stream_mut(orc_df11* d) { return d->stream; }

/* ===========================================================================
 * rANS tile codec (EntroPack section 3.6, appendix C.3; rANS after Duda 2013),
 * with MINE's k-tuple symbols (section 4, dtANS-LLM: "Pair" for k = 2).
 *
 * Alphabet: 4-bit codes -8..7 as values 0..15; a symbol is one code (k = 1) or the
 * codes of a lane's steps 2m and 2m+1 (k = 2), symbol = 16 * (c0 + 8) + (c1 + 8).
 * One frequency table per matrix with sum 2^prob_bits.  The matrix is flattened
 * row-major and cut into tiles of `tile` codes (the last may be short).  Inside a
 * tile, position q = 32*j + l belongs to lane l, step j.  State x lives in
 * [2^16, 2^32); payload words are 16 bits; the encoder starts every lane at
 * x = 2^16.
 * ========================================================================= */

/* reading: f_s = max(1, floor(M*c_s/n)) for present s; while the sum is short,
 * add 1 to the present symbol with the largest remainder M*c_s - f_s*n (ties to
 * the lower symbol); while it is over, take 1 from the present symbol with f_s > 1
 * and the smallest remainder (ties to the lower symbol).  Absent symbols get 0. */
int orc_rans_freqs_n(const uint64_t* counts, int nsym, int prob_bits, uint32_t* freqs) {
    const int64_t M = (int64_t)1 << prob_bits;
    uint64_t n = 0;
    int present = 0;
    for (int s = 0; s < nsym; ++s) {
        n += counts[s];
        present += counts[s] != 0;
    }
    memset(freqs, 0, (size_t)nsym * sizeof(uint32_t));
    if (n == 0) return 0;
    if (present > M) return -1;
    __int128* rem = (__int128*)calloc((size_t)nsym, sizeof(__int128));
    int64_t sum = 0;
    for (int s = 0; s < nsym; ++s) {
        if (!counts[s]) continue;
        int64_t f = (int64_t)(((unsigned __int128)M * counts[s]) / n);
        if (f < 1) f = 1;
        freqs[s] = (uint32_t)f;
        rem[s] = (__int128)M * (__int128)counts[s] - (__int128)f * (__int128)n;
        sum += f;
    }
    while (sum < M) {
        int best = -1;
        for (int s = 0; s < nsym; ++s)
            if (counts[s] && (best < 0 || rem[s] > rem[best])) best = s;
        freqs[best]++;
        rem[best] -= (__int128)n;
        ++sum;
    }
    while (sum > M) {
        int best = -1;
        for (int s = 0; s < nsym; ++s)
            if (counts[s] && freqs[s] > 1 && (best < 0 || rem[s] < rem[best])) best = s;
        if (best < 0) {
            free(rem);
            return -1;
        }
        freqs[best]--;
        rem[best] += (__int128)n;
        --sum;
    }
    free(rem);
    return present;
}

int orc_rans_freqs(const uint64_t counts[16], int prob_bits, uint32_t freqs[16]) {
    return orc_rans_freqs_n(counts, 16, prob_bits, freqs);
}

typedef struct {
    int64_t n;            /* codes */
    int prob_bits, tile, k, nsym;
    int64_t n_tiles;
    uint32_t freqs[256], cum[256];
    uint64_t counts[256];
    uint32_t* states;     /* n_tiles * 32: the decoder's initial (encoder's final) states */
    uint32_t* offsets;    /* n_tiles + 1: start of each tile's payload, in 16-bit words */
    uint16_t* payload;
    int64_t payload_words;
} orc_rans;

void orc_rans_free(orc_rans* r) {
    if (!r) return;
    free(r->states);
    free(r->offsets);
    free(r->payload);
    free(r);
}

static int64_t lane_steps(int64_t n_t, int l) { return n_t > l ? (n_t - l + 31) / 32 : 0; }

/* Symbol of lane l's symbol step m of a tile (codes at steps k*m .. k*m + k-1). */
static int tuple_symbol(const int8_t* tile_codes, int k, int64_t m, int l) {
    int s = 0;
    for (int i = 0; i < k; ++i) s = 16 * s + (tile_codes[32 * (k * m + i) + l] + 8);
    return s;
}

/* Encoder: each lane is encoded in reverse (last symbol step first); within a step
 * the lanes go 31 -> 0.  Before encoding s into x: while x >= f_s * 2^(32-prob_bits),
 * emit the low 16 bits and shift x right by 16 (with 2^16 <= x < 2^32 this is the
 * renormalisation bound ((2^16 >> b) << 16) * f_s).  Then
 * x = floor(x / f_s) * 2^b + (x mod f_s) + c_s.  Emitted words go on a stack; the
 * tile's payload is the stack read from the top, which is the order in which the
 * decoder asks for them.  With k = 2 every lane of every tile must hold an even
 * number of codes: tile and n multiples of 64. */
orc_rans* orc_rans_encode_k(const int8_t* codes, int64_t n, int prob_bits, int tile, int k) {
    if (n < 0 || prob_bits < 5 || prob_bits > 15 || tile < 32 || tile % 32) return NULL;
    if (k != 1 && k != 2) return NULL;
    if (k == 2 && (tile % 64 || n % 64)) return NULL;
    orc_rans* r = (orc_rans*)calloc(1, sizeof(orc_rans));
    r->n = n;
    r->prob_bits = prob_bits;
    r->tile = tile;
    r->k = k;
    r->nsym = k == 1 ? 16 : 256;
    for (int64_t i = 0; i < n; ++i) {
        if (codes[i] < -8 || codes[i] > 7) {
            orc_rans_free(r);
            return NULL;
        }
    }
    r->n_tiles = (n + tile - 1) / tile;
    for (int64_t t = 0; t < r->n_tiles; ++t) {
        const int64_t base = t * tile, n_t = (n - base < tile) ? n - base : tile;
        for (int l = 0; l < 32; ++l)
            for (int64_t m = 0; m < lane_steps(n_t, l) / k; ++m) r->counts[tuple_symbol(codes + base, k, m, l)]++;
    }
    if (orc_rans_freqs_n(r->counts, r->nsym, prob_bits, r->freqs) < 0) {
        orc_rans_free(r);
        return NULL;
    }
    for (int s = 0, c = 0; s < r->nsym; ++s) {
        r->cum[s] = (uint32_t)c;
        c += (int)r->freqs[s];
    }
    r->states = (uint32_t*)malloc(sizeof(uint32_t) * 32 * (size_t)(r->n_tiles > 0 ? r->n_tiles : 1));
    r->offsets = (uint32_t*)malloc(sizeof(uint32_t) * (size_t)(r->n_tiles + 1));
    r->payload = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(n > 0 ? n : 1)); /* <= 1 word per symbol */
    uint16_t* stack = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(tile));
    const uint64_t renorm_unit = (uint64_t)1 << (32 - prob_bits);
    int64_t words = 0;
    for (int64_t t = 0; t < r->n_tiles; ++t) {
        const int64_t base = t * tile;
        const int64_t n_t = (n - base < tile) ? n - base : tile;
        uint64_t x[32];
        for (int l = 0; l < 32; ++l) x[l] = 1u << 16;
        int64_t sp = 0;
        const int64_t steps = (n_t + 31) / 32 / k;
        for (int64_t m = steps - 1; m >= 0; --m) {
            for (int l = 31; l >= 0; --l) {
                if (m >= lane_steps(n_t, l) / k) continue;
                const int s = tuple_symbol(codes + base, k, m, l);
                const uint64_t f = r->freqs[s];
                while (x[l] >= f * renorm_unit) {
                    stack[sp++] = (uint16_t)(x[l] & 0xFFFF);
                    x[l] >>= 16;
                }
                x[l] = (x[l] / f << prob_bits) + (x[l] % f) + r->cum[s];
            }
        }
        for (int l = 0; l < 32; ++l) r->states[t * 32 + l] = (uint32_t)x[l];
        r->offsets[t] = (uint32_t)words;
        while (sp > 0) r->payload[words++] = stack[--sp];
    }
    r->offsets[r->n_tiles] = (uint32_t)words;
    r->payload_words = words;
    free(stack);
    return r;
}

orc_rans* orc_rans_encode(const int8_t* codes, int64_t n, int prob_bits, int tile) {
    return orc_rans_encode_k(codes, n, prob_bits, tile, 1);
}

/* Decoder: for symbol step m = 0.., lanes ascending: slot = x mod 2^b, s = the
 * symbol with c_s <= slot < c_s + f_s, x = f_s * (x >> b) + slot - c_s; if x < 2^16
 * then x = (x << 16) | next payload word; the symbol's codes go to the lane's
 * steps k*m .. k*m + k-1.  Also reports the lanes' final states (each must be
 * 2^16) and the words consumed (must be the tile's count).  Returns 0, -1 on a
 * corrupt stream, -2 if a final state or word count is off. */
int orc_rans_decode(const orc_rans* r, int8_t* out, uint32_t* final_states /* n_tiles*32 or NULL */) {
    const uint32_t M = 1u << r->prob_bits;
    const int k = r->k;
    int rc = 0;
    for (int64_t t = 0; t < r->n_tiles; ++t) {
        const int64_t base = t * r->tile;
        const int64_t n_t = (r->n - base < r->tile) ? r->n - base : r->tile;
        uint64_t x[32];
        for (int l = 0; l < 32; ++l) x[l] = r->states[t * 32 + l];
        int64_t wp = r->offsets[t];
        const int64_t wend = r->offsets[t + 1];
        const int64_t steps = (n_t + 31) / 32 / k;
        for (int64_t m = 0; m < steps; ++m) {
            for (int l = 0; l < 32; ++l) {
                if (m >= lane_steps(n_t, l) / k) continue;
                const uint32_t slot = (uint32_t)(x[l] & (M - 1));
                int s = -1;
                for (int q = 0; q < r->nsym; ++q)
                    if (r->freqs[q] && slot >= r->cum[q] && slot < r->cum[q] + r->freqs[q]) s = q;
                if (s < 0) return -1;
                x[l] = (uint64_t)r->freqs[s] * (x[l] >> r->prob_bits) + slot - r->cum[s];
                if (x[l] < (1u << 16)) {
                    if (wp >= wend) return -1;
                    x[l] = (x[l] << 16) | r->payload[wp++];
                }
                for (int i = k - 1, v = s; i >= 0; --i, v /= 16) out[base + 32 * (k * m + i) + l] = (int8_t)(v % 16 - 8);
            }
        }
        for (int l = 0; l < 32; ++l) {
            if (final_states) final_states[t * 32 + l] = (uint32_t)x[l];
            if (x[l] != (1u << 16)) rc = -2;
        }
        if (wp != wend) rc = -2;
    }
    return rc;
}

int64_t orc_rans_info(const orc_rans* r, int64_t* out /* 4 */) {
    out[0] = r->n;
    out[1] = r->n_tiles;
    out[2] = r->payload_words;
    out[3] = r->tile;
    return 0;
}
const uint32_t* orc_rans_freqs_of(const orc_rans* r) { return r->freqs; }
const uint64_t* orc_rans_counts_of(const orc_rans* r) { return r->counts; }
const uint32_t* orc_rans_states(const orc_rans* r) { return r->states; }
const uint32_t* orc_rans_offsets(const orc_rans* r) { return r->offsets; }
uint16_t* orc_rans_payload_mut(orc_rans* r) { return r->payload; }

/* FP4 E2M1 (the OCP Microscaling formats' 4-bit float; MINE lists FP4 among the
 * k-tuple data types, "Data Types", without fixing its value set): bit 3 the sign,
 * bits 1..2 the exponent field e with bias 1, bit 0 the mantissa bit m; e = 0 is
 * subnormal, m * 2^-1; otherwise (1 + m / 2) * 2^(e - 1).  No infinities or NaN. */
double orc_e2m1_value(int code) {
    const int sign = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
    const double mag = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return sign ? -mag : mag;
}

/* Dequantised weight w = value(code) * scale in FP32 (exact: a 4-bit integer, or an
 * E2M1 value of 2 significant bits, times an 11-bit significand), scale from group
 * floor(j / group) of row i.  values 0: the code is a signed integer in [-8, 7];
 * values 1: the code is an FP4 E2M1 pattern in [0, 15]. */
static float rans_weight(int8_t code, const uint16_t* scales, int64_t i, int64_t j, int64_t k_cols, int group,
                         int values) {
    const int64_t groups = (k_cols + group - 1) / group;
    const float v = values ? (float)orc_e2m1_value(code) : (float)code;
    return v * orc_f16_to_f32(scales[i * groups + j / group]);
}

/* BF16 (RNE) of the dequantised weights, the dense output of a decode. */
void orc_rans_dequant_bf16_v(const int8_t* codes, const uint16_t* scales, int64_t n_rows, int64_t k_cols,
                             int group, int values, uint16_t* out) {
    for (int64_t i = 0; i < n_rows; ++i)
        for (int64_t j = 0; j < k_cols; ++j)
            out[i * k_cols + j] =
                orc_f32_to_bf16_rne(rans_weight(codes[i * k_cols + j], scales, i, j, k_cols, group, values));
}
void orc_rans_dequant_bf16(const int8_t* codes, const uint16_t* scales, int64_t n_rows, int64_t k_cols,
                           int group, uint16_t* out) {
    orc_rans_dequant_bf16_v(codes, scales, n_rows, k_cols, group, 0, out);
}

/* ===========================================================================
 * GEMV in FP64: y[b,i] = sum_j w_ij * x_bj, summed in order j = 0..K-1, and
 * a[b,i] = sum_j |w_ij * x_bj| (the per-element error scale).
 * `rows` selects output rows (NULL = all); y and a are [batch, n_sel].
 * ========================================================================= */
void orc_gemv_bf16(const uint16_t* w, int64_t n_rows, int64_t k_cols, const uint16_t* x, int batch,
                   const int64_t* rows, int64_t n_sel, double* y, double* a) {
    const int64_t nr = rows ? n_sel : n_rows;
    for (int b = 0; b < batch; ++b) {
        for (int64_t r = 0; r < nr; ++r) {
            const int64_t i = rows ? rows[r] : r;
            double acc = 0.0, mag = 0.0;
            for (int64_t j = 0; j < k_cols; ++j) {
                const double p = orc_bf16_to_f64(w[i * k_cols + j]) * orc_bf16_to_f64(x[(int64_t)b * k_cols + j]);
                acc += p;
                mag += fabs(p);
            }
            y[(int64_t)b * nr + r] = acc;
            a[(int64_t)b * nr + r] = mag;
        }
    }
}

void orc_gemv_rans_v(const int8_t* codes, const uint16_t* scales, int64_t n_rows, int64_t k_cols, int group,
                     int values, const uint16_t* x, int batch, const int64_t* rows, int64_t n_sel, double* y,
                     double* a) {
    const int64_t nr = rows ? n_sel : n_rows;
    for (int b = 0; b < batch; ++b) {
        for (int64_t r = 0; r < nr; ++r) {
            const int64_t i = rows ? rows[r] : r;
            double acc = 0.0, mag = 0.0;
            for (int64_t j = 0; j < k_cols; ++j) {
                const double wv = (double)rans_weight(codes[i * k_cols + j], scales, i, j, k_cols, group, values);
                const double p = wv * orc_bf16_to_f64(x[(int64_t)b * k_cols + j]);
                acc += p;
                mag += fabs(p);
            }
            y[(int64_t)b * nr + r] = acc;
            a[(int64_t)b * nr + r] = mag;
        }
    }
}
void orc_gemv_rans(const int8_t* codes, const uint16_t* scales, int64_t n_rows, int64_t k_cols, int group,
                   const uint16_t* x, int batch, const int64_t* rows, int64_t n_sel, double* y, double* a) {
    orc_gemv_rans_v(codes, scales, n_rows, k_cols, group, 0, x, batch, rows, n_sel, y, a);
}

/* ===========================================================================
 * FP8 weights with a top-t decoding table and a sparse correction stream (MINE
 * section 4, "Escapes": the table keeps the t most frequent codes, always with
 * 0; any other value is coded as 0 and its true value goes to a correction
 * stream of one 32-bit record per escape).
 *
 * Readings (the pages fix the idea, not the record layout for this tile format):
 *  - codes are OCP FP8 E4M3 bytes; weight = fp32(value(code)) * r_i with an FP32
 *    scale per row; rows are padded to a multiple of 128 columns with code 0;
 *  - the table is code 0x00 and the t - 1 most frequent other codes present in
 *    the padded matrix (ties to the lower code), sorted by code; a symbol is a
 *    code's rank in it; a code outside the table is coded as symbol 0 (code 0x00);
 *  - symbols go through the tile codec above (one symbol per position, tiles of
 *    `tile` positions, position 32 j + l of a tile is lane l's step j);
 *  - tile t's records list its escapes by ascending position p: record =
 *    p | code << 16; rec_off[t] .. rec_off[t + 1] index them.
 * ========================================================================= */

/* Value of an E4M3 code: sign, 4 exponent bits (bias 7), 3 mantissa bits;
 * exponent field 0 holds the subnormals m/8 * 2^-6; S.1111.111 is NaN. */
float orc_e4m3_to_f32(uint8_t code) {
    const int s = code >> 7, e = (code >> 3) & 15, m = code & 7;
    if (e == 15 && m == 7) return NAN;
    const double v = e == 0 ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, e - 7);
    return (float)(s ? -v : v);
}

/* The top-t table of a code histogram: fills table[] (ascending codes) and
 * returns its size (<= t; t >= 1). */
int orc_fp8_table(const uint64_t counts[256], int t, uint8_t* table) {
    int chosen[256] = {0};
    chosen[0] = 1;
    int size = 1;
    while (size < t) {
        int best = -1;
        for (int c = 1; c < 256; ++c)
            if (!chosen[c] && counts[c] && (best < 0 || counts[c] > counts[best])) best = c;
        if (best < 0) break;
        chosen[best] = 1;
        ++size;
    }
    int n = 0;
    for (int c = 0; c < 256; ++c)
        if (chosen[c]) table[n++] = (uint8_t)c;
    return n;
}

typedef struct {
    int64_t n;                 /* positions (the padded layout, flattened) */
    int tsize;
    uint8_t table[256];
    int16_t rank[256];         /* code -> symbol, -1 outside the table */
    orc_rans* rans;            /* the symbol stream */
    uint32_t* rec_off;         /* n_tiles + 1 */
    uint32_t* records;
    int64_t n_records;
} orc_fp8;

void orc_fp8_free(orc_fp8* f) {
    if (!f) return;
    orc_rans_free(f->rans);
    free(f->rec_off);
    free(f->records);
    free(f);
}

/* Tile codec over a symbol array: as orc_rans_encode_k with k = 1, but the
 * symbols 0..nsym-1 are given (nsym <= 256). */
static orc_rans* rans_encode_symbols(const uint8_t* sym, int64_t n, int nsym, int prob_bits, int tile) {
    if (n < 0 || prob_bits < 5 || prob_bits > 15 || tile < 32 || tile % 32 || nsym < 1 || nsym > 256) return NULL;
    orc_rans* r = (orc_rans*)calloc(1, sizeof(orc_rans));
    r->n = n;
    r->prob_bits = prob_bits;
    r->tile = tile;
    r->k = 1;
    r->nsym = nsym;
    for (int64_t i = 0; i < n; ++i) r->counts[sym[i]]++;
    if (orc_rans_freqs_n(r->counts, nsym, prob_bits, r->freqs) < 0) {
        orc_rans_free(r);
        return NULL;
    }
    for (int s = 0, c = 0; s < nsym; ++s) {
        r->cum[s] = (uint32_t)c;
        c += (int)r->freqs[s];
    }
    r->n_tiles = (n + tile - 1) / tile;
    r->states = (uint32_t*)malloc(sizeof(uint32_t) * 32 * (size_t)(r->n_tiles > 0 ? r->n_tiles : 1));
    r->offsets = (uint32_t*)malloc(sizeof(uint32_t) * (size_t)(r->n_tiles + 1));
    r->payload = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(n > 0 ? n : 1));
    uint16_t* stack = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)tile);
    const uint64_t unit = (uint64_t)1 << (32 - prob_bits);
    int64_t words = 0;
    for (int64_t t = 0; t < r->n_tiles; ++t) {
        const int64_t base = t * tile, n_t = (n - base < tile) ? n - base : tile;
        uint64_t x[32];
        for (int l = 0; l < 32; ++l) x[l] = 1u << 16;
        int64_t sp = 0;
        for (int64_t m = (n_t + 31) / 32 - 1; m >= 0; --m)
            for (int l = 31; l >= 0; --l) {
                if (32 * m + l >= n_t) continue;
                const int s = sym[base + 32 * m + l];
                const uint64_t f = r->freqs[s];
                while (x[l] >= f * unit) {
                    stack[sp++] = (uint16_t)(x[l] & 0xFFFF);
                    x[l] >>= 16;
                }
                x[l] = (x[l] / f << prob_bits) + (x[l] % f) + r->cum[s];
            }
        for (int l = 0; l < 32; ++l) r->states[t * 32 + l] = (uint32_t)x[l];
        r->offsets[t] = (uint32_t)words;
        while (sp > 0) r->payload[words++] = stack[--sp];
    }
    r->offsets[r->n_tiles] = (uint32_t)words;
    r->payload_words = words;
    free(stack);
    return r;
}

/* Encode the padded FP8 layout codes[n] with a table of at most t codes. */
orc_fp8* orc_fp8_encode(const uint8_t* codes, int64_t n, int t, int prob_bits, int tile) {
    if (n < 0 || t < 1 || t > 256) return NULL;
    for (int64_t i = 0; i < n; ++i)
        if ((codes[i] & 0x7F) == 0x7F) return NULL; /* NaN */
    orc_fp8* f = (orc_fp8*)calloc(1, sizeof(orc_fp8));
    f->n = n;
    uint64_t counts[256] = {0};
    for (int64_t i = 0; i < n; ++i) counts[codes[i]]++;
    f->tsize = orc_fp8_table(counts, t, f->table);
    for (int c = 0; c < 256; ++c) f->rank[c] = -1;
    for (int s = 0; s < f->tsize; ++s) f->rank[f->table[s]] = (int16_t)s;
    uint8_t* sym = (uint8_t*)malloc((size_t)(n > 0 ? n : 1));
    for (int64_t i = 0; i < n; ++i) sym[i] = f->rank[codes[i]] >= 0 ? (uint8_t)f->rank[codes[i]] : 0;
    f->rans = rans_encode_symbols(sym, n, f->tsize, prob_bits, tile);
    free(sym);
    if (!f->rans) {
        orc_fp8_free(f);
        return NULL;
    }
    const int64_t nt = f->rans->n_tiles;
    f->rec_off = (uint32_t*)malloc(sizeof(uint32_t) * (size_t)(nt + 1));
    int64_t ne = 0;
    for (int64_t i = 0; i < n; ++i) ne += f->rank[codes[i]] < 0;
    f->records = (uint32_t*)malloc(sizeof(uint32_t) * (size_t)(ne > 0 ? ne : 1));
    f->n_records = 0;
    for (int64_t tt = 0; tt < nt; ++tt) {
        f->rec_off[tt] = (uint32_t)f->n_records;
        const int64_t base = tt * tile, n_t = (n - base < tile) ? n - base : tile;
        for (int64_t p = 0; p < n_t; ++p)
            if (f->rank[codes[base + p]] < 0) f->records[f->n_records++] = (uint32_t)p | ((uint32_t)codes[base + p] << 16);
    }
    f->rec_off[nt] = (uint32_t)f->n_records;
    return f;
}

/* Decode back to codes: the tile codec's symbols through the table, then each
 * record's code at its position.  Returns the tile codec's status (0 ok). */
int orc_fp8_decode(const orc_fp8* f, uint8_t* codes) {
    const orc_rans* r = f->rans;
    const uint32_t M = 1u << r->prob_bits;
    int rc = 0;
    for (int64_t t = 0; t < r->n_tiles; ++t) {
        const int64_t base = t * r->tile, n_t = (r->n - base < r->tile) ? r->n - base : r->tile;
        uint64_t x[32];
        for (int l = 0; l < 32; ++l) x[l] = r->states[t * 32 + l];
        int64_t wp = r->offsets[t];
        const int64_t wend = r->offsets[t + 1];
        for (int64_t m = 0; m < (n_t + 31) / 32; ++m)
            for (int l = 0; l < 32; ++l) {
                if (32 * m + l >= n_t) continue;
                const uint32_t slot = (uint32_t)(x[l] & (M - 1));
                int s = -1;
                for (int q = 0; q < r->nsym; ++q)
                    if (r->freqs[q] && slot >= r->cum[q] && slot < r->cum[q] + r->freqs[q]) s = q;
                if (s < 0) return -1;
                x[l] = (uint64_t)r->freqs[s] * (x[l] >> r->prob_bits) + slot - r->cum[s];
                if (x[l] < (1u << 16)) {
                    if (wp >= wend) return -1;
                    x[l] = (x[l] << 16) | r->payload[wp++];
                }
                codes[base + 32 * m + l] = f->table[s];
            }
        for (int l = 0; l < 32; ++l)
            if (x[l] != (1u << 16)) rc = -2;
        if (wp != wend) rc = -2;
        for (uint32_t e = f->rec_off[t]; e < f->rec_off[t + 1]; ++e) {
            const uint32_t p = f->records[e] & 0xFFFFu;
            if ((int64_t)p >= n_t) return -1;
            codes[base + p] = (uint8_t)(f->records[e] >> 16);
        }
    }
    return rc;
}

int64_t orc_fp8_info(const orc_fp8* f, int64_t* out /* 6 */) {
    out[0] = f->n;
    out[1] = f->rans->n_tiles;
    out[2] = f->rans->payload_words;
    out[3] = f->rans->tile;
    out[4] = f->tsize;
    out[5] = f->n_records;
    return 0;
}
const uint8_t* orc_fp8_table_of(const orc_fp8* f) { return f->table; }
const uint32_t* orc_fp8_freqs_of(const orc_fp8* f) { return f->rans->freqs; }
const uint64_t* orc_fp8_counts_of(const orc_fp8* f) { return f->rans->counts; }
const uint32_t* orc_fp8_states(const orc_fp8* f) { return f->rans->states; }
const uint32_t* orc_fp8_offsets(const orc_fp8* f) { return f->rans->offsets; }
uint16_t* orc_fp8_payload_mut(orc_fp8* f) { return f->rans->payload; }
const uint32_t* orc_fp8_rec_off(const orc_fp8* f) { return f->rec_off; }
const uint32_t* orc_fp8_records(const orc_fp8* f) { return f->records; }

/* Dense BF16 of FP8 codes [n_rows, k_cols] with FP32 row scales:
 * bf16(fp32(value(code) * r_i)). */
void orc_fp8_dequant_bf16(const uint8_t* codes, const float* r, int64_t n_rows, int64_t k_cols, uint16_t* out) {
    for (int64_t i = 0; i < n_rows; ++i)
        for (int64_t j = 0; j < k_cols; ++j)
            out[i * k_cols + j] = orc_f32_to_bf16_rne(orc_e4m3_to_f32(codes[i * k_cols + j]) * r[i]);
}

/* FP64 y[b, i] = sum_j value(code_ij) r_i x_bj and a = sum |...|, in index order. */
void orc_gemv_fp8(const uint8_t* codes, const float* r, int64_t n_rows, int64_t k_cols, const uint16_t* x,
                  int batch, const int64_t* rows, int64_t n_sel, double* y, double* a) {
    const int64_t nr = rows ? n_sel : n_rows;
    for (int b = 0; b < batch; ++b)
        for (int64_t q = 0; q < nr; ++q) {
            const int64_t i = rows ? rows[q] : q;
            double acc = 0.0, mag = 0.0;
            for (int64_t j = 0; j < k_cols; ++j) {
                const double p = (double)orc_e4m3_to_f32(codes[i * k_cols + j]) * (double)r[i] *
                                 orc_bf16_to_f64(x[(int64_t)b * k_cols + j]);
                acc += p;
                mag += fabs(p);
            }
            y[(int64_t)b * nr + q] = acc;
            a[(int64_t)b * nr + q] = mag;
        }
}

/* ===========================================================================
 * E8 lattice fields, EntroPack sections 3.2 (row-normalised lattice
 * representation), 3.3 (coset-conditioned model), 3.6 (tiles), 3.7 (GPU
 * reconstruction) and appendix A.3 (parity reduction).
 *
 * Weights go in blocks of 8 along a row; block p of row i stands for
 * w = s * r_i * p with p in E8 = D8 u (D8 + h), h = (1/2, ..., 1/2) and
 * D8 = { z in Z^8 : z_1 + ... + z_8 even }.  A point is given doubled, q = 2p
 * (integers, all eight with the same parity).
 *
 * Readings (the pages name the fields, not their formulas):
 *  - coset c = q_1 mod 2 (0: D8, 1: D8 + h); coordinates z_j = (q_j - c) / 2;
 *  - parity reduction: the eighth coordinate is coded as m with
 *    z_8 = 2 m + ((z_1 + ... + z_7) mod 2), so every coded (c, z_1..z_7, m) is a
 *    lattice point and every lattice point has exactly one code;
 *  - 17 categorical tables: table 0 for c, table 1 + 8 c + f for field f of
 *    (z_1, ..., z_7, m) under coset c; field values are offset by 16 (z_j in
 *    -16..15, m in -8..7, alphabet 0..31);
 *  - reconstruction in FP32: g_i = s * r_i, w = (q * g_i) * 0.5, then BF16 (RNE).
 *
 * rANS as in the tile codec above (states in [2^16, 2^32), 16-bit words, one
 * table per field with sum 2^prob_bits): tiles of `tile` vectors, lane l owns the
 * tile's vectors l, l + 32, ...; vector j of a lane is nine symbol steps
 * 9 j .. 9 j + 8 (c first), and at each step the lanes take words in lane order.
 * ========================================================================= */
#define E8_FIELDS 9
#define E8_TABLES 17
#define E8_ALPHA 32

/* Fields of a doubled point q[8] (c, z_1 + 16, ..., z_7 + 16, m + 16); -1 if q is
 * not in 2 E8 or a field is out of range. */
int orc_e8_fields(const int8_t* q, int* fields) {
    const int c = q[0] & 1;
    int z[8], sum7 = 0;
    for (int j = 0; j < 8; ++j) {
        if ((q[j] & 1) != c) return -1;
        z[j] = (q[j] - c) / 2;
    }
    int total = 0;
    for (int j = 0; j < 8; ++j) total += z[j];
    if (total % 2) return -1; /* z must be in D8 */
    for (int j = 0; j < 7; ++j) sum7 += z[j];
    const int par = ((sum7 % 2) + 2) % 2;
    const int m = (z[7] - par) / 2; /* exact: z_8 - par is even */
    fields[0] = c;
    for (int j = 0; j < 7; ++j) {
        if (z[j] < -16 || z[j] > 15) return -1;
        fields[1 + j] = z[j] + 16;
    }
    if (m < -8 || m > 7) return -1;
    fields[8] = m + 16;
    return 0;
}

/* The doubled point of a field vector (inverse of orc_e8_fields). */
void orc_e8_point(const int* fields, int8_t* q) {
    const int c = fields[0];
    int z[8], sum7 = 0;
    for (int j = 0; j < 7; ++j) {
        z[j] = fields[1 + j] - 16;
        sum7 += z[j];
    }
    const int par = ((sum7 % 2) + 2) % 2;
    z[7] = 2 * (fields[8] - 16) + par;
    for (int j = 0; j < 8; ++j) q[j] = (int8_t)(2 * z[j] + c);
}

static int e8_table(int f, int c) { return f == 0 ? 0 : 1 + 8 * c + (f - 1); }

typedef struct {
    int64_t n_vec;
    int prob_bits, tile;
    int64_t n_tiles;
    uint64_t counts[E8_TABLES][E8_ALPHA];
    uint32_t freqs[E8_TABLES][E8_ALPHA], cum[E8_TABLES][E8_ALPHA];
    uint32_t* states;
    uint32_t* offsets;
    uint16_t* payload;
    int64_t payload_words;
} orc_e8;

void orc_e8_free(orc_e8* e) {
    if (!e) return;
    free(e->states);
    free(e->offsets);
    free(e->payload);
    free(e);
}

/* Encode n_vec doubled points q[n_vec][8]; NULL if a point is invalid. */
orc_e8* orc_e8_encode(const int8_t* q, int64_t n_vec, int prob_bits, int tile) {
    if (n_vec < 0 || prob_bits < 5 || prob_bits > 15 || tile < 32 || tile % 32) return NULL;
    orc_e8* e = (orc_e8*)calloc(1, sizeof(orc_e8));
    e->n_vec = n_vec;
    e->prob_bits = prob_bits;
    e->tile = tile;
    int* fields = (int*)malloc(sizeof(int) * E8_FIELDS * (size_t)(n_vec > 0 ? n_vec : 1));
    for (int64_t v = 0; v < n_vec; ++v) {
        if (orc_e8_fields(q + 8 * v, fields + E8_FIELDS * v) < 0) {
            free(fields);
            orc_e8_free(e);
            return NULL;
        }
        const int* fv = fields + E8_FIELDS * v;
        for (int f = 0; f < E8_FIELDS; ++f) e->counts[e8_table(f, fv[0])][fv[f]]++;
    }
    for (int t = 0; t < E8_TABLES; ++t) {
        if (orc_rans_freqs_n(e->counts[t], E8_ALPHA, prob_bits, e->freqs[t]) < 0) {
            free(fields);
            orc_e8_free(e);
            return NULL;
        }
        for (int s = 0, c = 0; s < E8_ALPHA; ++s) {
            e->cum[t][s] = (uint32_t)c;
            c += (int)e->freqs[t][s];
        }
    }
    e->n_tiles = (n_vec + tile - 1) / tile;
    e->states = (uint32_t*)malloc(sizeof(uint32_t) * 32 * (size_t)(e->n_tiles > 0 ? e->n_tiles : 1));
    e->offsets = (uint32_t*)malloc(sizeof(uint32_t) * (size_t)(e->n_tiles + 1));
    e->payload = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(E8_FIELDS * n_vec + 1));
    uint16_t* stack = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(E8_FIELDS * tile));
    const uint64_t renorm_unit = (uint64_t)1 << (32 - prob_bits);
    int64_t words = 0;
    for (int64_t t = 0; t < e->n_tiles; ++t) {
        const int64_t base = t * tile, n_t = (n_vec - base < tile) ? n_vec - base : tile;
        uint64_t x[32];
        for (int l = 0; l < 32; ++l) x[l] = 1u << 16;
        int64_t sp = 0;
        for (int64_t j = (n_t + 31) / 32 - 1; j >= 0; --j) {
            for (int f = E8_FIELDS - 1; f >= 0; --f) {
                for (int l = 31; l >= 0; --l) {
                    const int64_t v = base + 32 * j + l;
                    if (32 * j + l >= n_t) continue;
                    const int* fv = fields + E8_FIELDS * v;
                    const int tb = e8_table(f, fv[0]), s = fv[f];
                    const uint64_t fr = e->freqs[tb][s];
                    while (x[l] >= fr * renorm_unit) {
                        stack[sp++] = (uint16_t)(x[l] & 0xFFFF);
                        x[l] >>= 16;
                    }
                    x[l] = (x[l] / fr << prob_bits) + (x[l] % fr) + e->cum[tb][s];
                }
            }
        }
        for (int l = 0; l < 32; ++l) e->states[t * 32 + l] = (uint32_t)x[l];
        e->offsets[t] = (uint32_t)words;
        while (sp > 0) e->payload[words++] = stack[--sp];
    }
    e->offsets[e->n_tiles] = (uint32_t)words;
    e->payload_words = words;
    free(stack);
    free(fields);
    return e;
}

/* Decode to doubled points q_out[n_vec][8].  Returns 0, -1 on a corrupt stream, -2
 * if a final state is not 2^16 or a tile's words are not used up. */
int orc_e8_decode(const orc_e8* e, int8_t* q_out, uint32_t* final_states) {
    const uint32_t M = 1u << e->prob_bits;
    int rc = 0;
    for (int64_t t = 0; t < e->n_tiles; ++t) {
        const int64_t base = t * e->tile, n_t = (e->n_vec - base < e->tile) ? e->n_vec - base : e->tile;
        uint64_t x[32];
        int fv[32][E8_FIELDS];
        for (int l = 0; l < 32; ++l) x[l] = e->states[t * 32 + l];
        int64_t wp = e->offsets[t];
        const int64_t wend = e->offsets[t + 1];
        for (int64_t j = 0; j < (n_t + 31) / 32; ++j) {
            for (int f = 0; f < E8_FIELDS; ++f) {
                for (int l = 0; l < 32; ++l) {
                    if (32 * j + l >= n_t) continue;
                    const int tb = e8_table(f, f == 0 ? 0 : fv[l][0]);
                    const uint32_t slot = (uint32_t)(x[l] & (M - 1));
                    int s = -1;
                    for (int k = 0; k < E8_ALPHA; ++k)
                        if (e->freqs[tb][k] && slot >= e->cum[tb][k] && slot < e->cum[tb][k] + e->freqs[tb][k]) s = k;
                    if (s < 0) return -1;
                    x[l] = (uint64_t)e->freqs[tb][s] * (x[l] >> e->prob_bits) + slot - e->cum[tb][s];
                    if (x[l] < (1u << 16)) {
                        if (wp >= wend) return -1;
                        x[l] = (x[l] << 16) | e->payload[wp++];
                    }
                    fv[l][f] = s;
                }
            }
            for (int l = 0; l < 32; ++l)
                if (32 * j + l < n_t) orc_e8_point(fv[l], q_out + 8 * (base + 32 * j + l));
        }
        for (int l = 0; l < 32; ++l) {
            if (final_states) final_states[t * 32 + l] = (uint32_t)x[l];
            if (x[l] != (1u << 16)) rc = -2;
        }
        if (wp != wend) rc = -2;
    }
    return rc;
}

int64_t orc_e8_info(const orc_e8* e, int64_t* out /* 4 */) {
    out[0] = e->n_vec;
    out[1] = e->n_tiles;
    out[2] = e->payload_words;
    out[3] = e->tile;
    return 0;
}
const uint32_t* orc_e8_freqs_of(const orc_e8* e) { return &e->freqs[0][0]; }
const uint64_t* orc_e8_counts_of(const orc_e8* e) { return &e->counts[0][0]; }
const uint32_t* orc_e8_states(const orc_e8* e) { return e->states; }
const uint32_t* orc_e8_offsets(const orc_e8* e) { return e->offsets; }
uint16_t* orc_e8_payload_mut(orc_e8* e) { return e->payload; }

/* The E8 reconstruction v = fp32(fp32(q) * g_i) * 0.5 with g_i = fp32(s * r_i), written
 * in the requested dtype (EntroPack section 3.7: floating-point or integer output,
 * FP8 and INT8 included): 0 = BF16 (u16 out, RNE), 1 = FP8 E4M3 (u8 out, RNE,
 * saturating), 2 = INT8 (RNE, saturating). */
void orc_e8_reconstruct_as(const int8_t* q, int64_t n_rows, int64_t k_cols, float s, const float* r, int dtype,
                           void* out) {
    for (int64_t i = 0; i < n_rows; ++i) {
        const float g = s * r[i];
        for (int64_t j = 0; j < k_cols; ++j) {
            const float v = ((float)q[i * k_cols + j] * g) * 0.5f;
            const int64_t at = i * k_cols + j;
            if (dtype == 0) ((uint16_t*)out)[at] = orc_f32_to_bf16_rne(v);
            else if (dtype == 1) ((uint8_t*)out)[at] = orc_f32_to_e4m3_satfinite(v);
            else ((int8_t*)out)[at] = orc_f32_to_s8_rne_sat(v);
        }
    }
}

/* BF16 weights of doubled points q [n_rows, k_cols] (k_cols % 8 == 0): row i's
 * factor g_i = fp32(s * r_i), w = bf16(fp32(fp32(q) * g_i) * 0.5). */
void orc_e8_reconstruct_bf16(const int8_t* q, int64_t n_rows, int64_t k_cols, float s, const float* r,
                             uint16_t* out) {
    for (int64_t i = 0; i < n_rows; ++i) {
        const float g = s * r[i];
        for (int64_t j = 0; j < k_cols; ++j) {
            const float v = (float)q[i * k_cols + j] * g;
            out[i * k_cols + j] = orc_f32_to_bf16_rne(v * 0.5f);
        }
    }
}

/* ===========================================================================
 * BF16 exponents through rANS tiles with a top-t table and escape records
 * (MINE section 4: dtANS-LLM's BF16 handling -- the exponent is entropy-coded,
 * sign and mantissa are kept as one plain byte; "Escapes": the table holds the t
 * most frequent values and always 0, a value outside it is coded as 0 and listed
 * in a sparse correction stream; "Pair" symbols of two values when t^2 <= M;
 * "Tuning t": the t with the smallest size bound, cross-entropy of the stream plus
 * a 4-byte record per escape).
 *
 * Readings:
 *  - the coded value is the exponent field e = bits 7..14 of the BF16 pattern;
 *    the plain byte is sign << 7 | mantissa (bits 15 and 0..6);
 *  - the table is exponent 0 and the t - 1 most frequent other exponents present
 *    (ties to the lower exponent), sorted ascending (the rule of orc_fp8_table);
 *    an exponent's symbol value is its rank there, and an escaped exponent is
 *    coded as rank 0 (exponent 0);
 *  - positions are those of the padded layout (rows of k_pad columns, zero
 *    weights in the padding), flattened, in tiles of `tile` positions; position
 *    32 j + l of a tile is lane l's step j (as the tile codec above);
 *  - k = 1: one symbol per lane step; k = 2: the symbol of lane steps 2 m and
 *    2 m + 1 is rank(e_2m) * tsize + rank(e_2m+1) (tile and n multiples of 64);
 *  - one frequency table over the tsize^k symbol values (orc_rans_freqs_n),
 *    states and payload words as the tile codec above;
 *  - tile t's records list its escapes by ascending position p: p | e << 16;
 *  - size bound of a table size t: sum over the stream's symbols of
 *    log2(2^prob_bits / f_s) bits plus 32 bits per escape; the automatic t is the
 *    smallest t in 1..t_max with the least bound.
 * ========================================================================= */
typedef struct {
    int64_t n;                 /* positions */
    int k, tsize, prob_bits, tile, nsym;
    uint8_t table[256];
    int16_t rank[256];
    uint32_t* freqs;           /* nsym */
    uint32_t* cum;
    uint64_t* counts;
    int64_t n_tiles;
    uint32_t* states;          /* n_tiles * 32 */
    uint32_t* offsets;         /* n_tiles + 1 */
    uint16_t* payload;
    int64_t payload_words;
    uint32_t* rec_off;         /* n_tiles + 1 */
    uint32_t* records;
    int64_t n_records;
    uint8_t* sm;               /* n plain bytes: sign << 7 | mantissa */
} orc_expx;

void orc_expx_free(orc_expx* f) {
    if (!f) return;
    free(f->freqs);
    free(f->cum);
    free(f->counts);
    free(f->states);
    free(f->offsets);
    free(f->payload);
    free(f->rec_off);
    free(f->records);
    free(f->sm);
    free(f);
}

static int expx_field(uint16_t w) { return (w >> 7) & 0xFF; }

/* The symbol of lane l's symbol step m in the tile starting at `base` (n_t
 * positions), given the rank of every position's exponent (escapes already 0). */
static int expx_symbol(const uint8_t* rk, int64_t base, int k, int tsize, int64_t m, int l) {
    int s = 0;
    for (int i = 0; i < k; ++i) s = s * tsize + rk[base + 32 * (k * m + i) + l];
    return s;
}

/* Ranks of every position under the table of size t built from `counts`; the
 * number of escapes goes to *n_esc.  Returns the table size. */
static int expx_ranks(const uint16_t* w, int64_t n, const uint64_t counts[256], int t, uint8_t* table, int16_t* rank,
                      uint8_t* rk, int64_t* n_esc) {
    const int tsize = orc_fp8_table(counts, t, table);
    for (int e = 0; e < 256; ++e) rank[e] = -1;
    for (int s = 0; s < tsize; ++s) rank[table[s]] = (int16_t)s;
    int64_t ne = 0;
    for (int64_t i = 0; i < n; ++i) {
        const int r = rank[expx_field(w[i])];
        rk[i] = (uint8_t)(r < 0 ? 0 : r);
        ne += r < 0;
    }
    *n_esc = ne;
    return tsize;
}

/* Histogram of the symbol stream (nsym values). */
static void expx_histogram(const uint8_t* rk, int64_t n, int k, int tsize, int tile, uint64_t* counts, int nsym) {
    memset(counts, 0, sizeof(uint64_t) * (size_t)nsym);
    for (int64_t base = 0; base < n; base += tile) {
        const int64_t n_t = (n - base < tile) ? n - base : tile;
        for (int l = 0; l < 32; ++l)
            for (int64_t m = 0; m < lane_steps(n_t, l) / k; ++m) counts[expx_symbol(rk, base, k, tsize, m, l)]++;
    }
}

/* Size bound in bits of table size t (k, prob_bits fixed); -1 when the table
 * cannot hold the symbol values (tsize^k > 2^prob_bits). */
double orc_expx_bound(const uint16_t* w, int64_t n, int k, int t, int prob_bits, int tile) {
    uint64_t cnt[256] = {0};
    for (int64_t i = 0; i < n; ++i) cnt[expx_field(w[i])]++;
    uint8_t table[256];
    int16_t rank[256];
    uint8_t* rk = (uint8_t*)malloc((size_t)(n > 0 ? n : 1));
    int64_t ne = 0;
    const int tsize = expx_ranks(w, n, cnt, t, table, rank, rk, &ne);
    const int nsym = k == 1 ? tsize : tsize * tsize;
    if (nsym > (1 << prob_bits)) {
        free(rk);
        return -1.0;
    }
    uint64_t* counts = (uint64_t*)calloc((size_t)nsym, sizeof(uint64_t));
    uint32_t* freqs = (uint32_t*)calloc((size_t)nsym, sizeof(uint32_t));
    expx_histogram(rk, n, k, tsize, tile, counts, nsym);
    double bits = 0.0;
    if (orc_rans_freqs_n(counts, nsym, prob_bits, freqs) >= 0)
        for (int s = 0; s < nsym; ++s)
            if (counts[s]) bits += (double)counts[s] * ((double)prob_bits - log2((double)freqs[s]));
    free(counts);
    free(freqs);
    free(rk);
    return bits + 32.0 * (double)ne;
}

/* The smallest t in 1..t_max with the least bound (t_max capped where tsize^k
 * would exceed the table). */
int orc_expx_choose_t(const uint16_t* w, int64_t n, int k, int t_max, int prob_bits, int tile) {
    int best = 1;
    double best_bits = -1.0;
    for (int t = 1; t <= t_max && t <= 256; ++t) {
        const double b = orc_expx_bound(w, n, k, t, prob_bits, tile);
        if (b < 0) break;
        if (best_bits < 0 || b < best_bits) {
            best_bits = b;
            best = t;
        }
    }
    return best;
}

/* Encode BF16 patterns w[n] (the padded layout, flattened). */
orc_expx* orc_expx_encode(const uint16_t* w, int64_t n, int t, int prob_bits, int tile, int k) {
    if (n < 0 || t < 1 || t > 256 || prob_bits < 5 || prob_bits > 15 || tile < 32 || tile % 32) return NULL;
    if (k != 1 && k != 2) return NULL;
    if (k == 2 && (tile % 64 || n % 64)) return NULL;
    orc_expx* f = (orc_expx*)calloc(1, sizeof(orc_expx));
    f->n = n;
    f->k = k;
    f->prob_bits = prob_bits;
    f->tile = tile;
    uint64_t cnt[256] = {0};
    for (int64_t i = 0; i < n; ++i) cnt[expx_field(w[i])]++;
    uint8_t* rk = (uint8_t*)malloc((size_t)(n > 0 ? n : 1));
    int64_t ne = 0;
    f->tsize = expx_ranks(w, n, cnt, t, f->table, f->rank, rk, &ne);
    f->nsym = k == 1 ? f->tsize : f->tsize * f->tsize;
    if (f->nsym > (1 << prob_bits)) {
        free(rk);
        orc_expx_free(f);
        return NULL;
    }
    f->counts = (uint64_t*)calloc((size_t)f->nsym, sizeof(uint64_t));
    f->freqs = (uint32_t*)calloc((size_t)f->nsym, sizeof(uint32_t));
    f->cum = (uint32_t*)calloc((size_t)f->nsym, sizeof(uint32_t));
    expx_histogram(rk, n, k, f->tsize, tile, f->counts, f->nsym);
    if (orc_rans_freqs_n(f->counts, f->nsym, prob_bits, f->freqs) < 0) {
        free(rk);
        orc_expx_free(f);
        return NULL;
    }
    for (int s = 0, c = 0; s < f->nsym; ++s) {
        f->cum[s] = (uint32_t)c;
        c += (int)f->freqs[s];
    }
    /* the symbol stream: each lane in reverse, lanes 31 -> 0 within a step (as
     * orc_rans_encode_k) */
    f->n_tiles = (n + tile - 1) / tile;
    f->states = (uint32_t*)malloc(sizeof(uint32_t) * 32 * (size_t)(f->n_tiles > 0 ? f->n_tiles : 1));
    f->offsets = (uint32_t*)malloc(sizeof(uint32_t) * (size_t)(f->n_tiles + 1));
    f->payload = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(n > 0 ? n : 1));
    uint16_t* stack = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)tile);
    const uint64_t unit = (uint64_t)1 << (32 - prob_bits);
    int64_t words = 0;
    for (int64_t tt = 0; tt < f->n_tiles; ++tt) {
        const int64_t base = tt * tile, n_t = (n - base < tile) ? n - base : tile;
        uint64_t x[32];
        for (int l = 0; l < 32; ++l) x[l] = 1u << 16;
        int64_t sp = 0;
        for (int64_t m = (n_t + 31) / 32 / k - 1; m >= 0; --m)
            for (int l = 31; l >= 0; --l) {
                if (m >= lane_steps(n_t, l) / k) continue;
                const int s = expx_symbol(rk, base, k, f->tsize, m, l);
                const uint64_t fs = f->freqs[s];
                while (x[l] >= fs * unit) {
                    stack[sp++] = (uint16_t)(x[l] & 0xFFFF);
                    x[l] >>= 16;
                }
                x[l] = (x[l] / fs << prob_bits) + (x[l] % fs) + f->cum[s];
            }
        for (int l = 0; l < 32; ++l) f->states[tt * 32 + l] = (uint32_t)x[l];
        f->offsets[tt] = (uint32_t)words;
        while (sp > 0) f->payload[words++] = stack[--sp];
    }
    f->offsets[f->n_tiles] = (uint32_t)words;
    f->payload_words = words;
    free(stack);
    free(rk);
    /* escapes and plain bytes */
    f->rec_off = (uint32_t*)malloc(sizeof(uint32_t) * (size_t)(f->n_tiles + 1));
    f->records = (uint32_t*)malloc(sizeof(uint32_t) * (size_t)(ne > 0 ? ne : 1));
    f->sm = (uint8_t*)malloc((size_t)(n > 0 ? n : 1));
    for (int64_t tt = 0; tt < f->n_tiles; ++tt) {
        f->rec_off[tt] = (uint32_t)f->n_records;
        const int64_t base = tt * tile, n_t = (n - base < tile) ? n - base : tile;
        for (int64_t p = 0; p < n_t; ++p) {
            const int e = expx_field(w[base + p]);
            if (f->rank[e] < 0) f->records[f->n_records++] = (uint32_t)p | ((uint32_t)e << 16);
        }
    }
    f->rec_off[f->n_tiles] = (uint32_t)f->n_records;
    for (int64_t i = 0; i < n; ++i) f->sm[i] = (uint8_t)(((w[i] >> 8) & 0x80) | (w[i] & 0x7F));
    return f;
}

/* Decode back to BF16 patterns: symbols through the table (ranks to exponents),
 * each record's exponent at its position, then sign | exponent | mantissa.
 * Returns 0, -1 on a corrupt stream, -2 if a final state or word count is off. */
int orc_expx_decode(const orc_expx* f, uint16_t* out) {
    const uint32_t M = 1u << f->prob_bits;
    const int k = f->k;
    int rc = 0;
    uint8_t* ex = (uint8_t*)malloc((size_t)(f->n > 0 ? f->n : 1));
    for (int64_t t = 0; t < f->n_tiles; ++t) {
        const int64_t base = t * f->tile, n_t = (f->n - base < f->tile) ? f->n - base : f->tile;
        uint64_t x[32];
        for (int l = 0; l < 32; ++l) x[l] = f->states[t * 32 + l];
        int64_t wp = f->offsets[t];
        const int64_t wend = f->offsets[t + 1];
        for (int64_t m = 0; m < (n_t + 31) / 32 / k; ++m)
            for (int l = 0; l < 32; ++l) {
                if (m >= lane_steps(n_t, l) / k) continue;
                const uint32_t slot = (uint32_t)(x[l] & (M - 1));
                int s = -1;
                for (int q = 0; q < f->nsym; ++q)
                    if (f->freqs[q] && slot >= f->cum[q] && slot < f->cum[q] + f->freqs[q]) s = q;
                if (s < 0) {
                    free(ex);
                    return -1;
                }
                x[l] = (uint64_t)f->freqs[s] * (x[l] >> f->prob_bits) + slot - f->cum[s];
                if (x[l] < (1u << 16)) {
                    if (wp >= wend) {
                        free(ex);
                        return -1;
                    }
                    x[l] = (x[l] << 16) | f->payload[wp++];
                }
                for (int i = k - 1, v = s; i >= 0; --i, v /= f->tsize)
                    ex[base + 32 * (k * m + i) + l] = f->table[v % f->tsize];
            }
        for (int l = 0; l < 32; ++l)
            if (x[l] != (1u << 16)) rc = -2;
        if (wp != wend) rc = -2;
        for (uint32_t e = f->rec_off[t]; e < f->rec_off[t + 1]; ++e) {
            const uint32_t p = f->records[e] & 0xFFFFu;
            if ((int64_t)p >= n_t) {
                free(ex);
                return -1;
            }
            ex[base + p] = (uint8_t)(f->records[e] >> 16);
        }
    }
    for (int64_t i = 0; i < f->n; ++i)
        out[i] = (uint16_t)(((uint16_t)(f->sm[i] & 0x80) << 8) | ((uint16_t)ex[i] << 7) | (f->sm[i] & 0x7F));
    free(ex);
    return rc;
}

int64_t orc_expx_info(const orc_expx* f, int64_t* out /* 8 */) {
    out[0] = f->n;
    out[1] = f->n_tiles;
    out[2] = f->payload_words;
    out[3] = f->tile;
    out[4] = f->tsize;
    out[5] = f->n_records;
    out[6] = f->nsym;
    out[7] = f->k;
    return 0;
}
const uint8_t* orc_expx_table_of(const orc_expx* f) { return f->table; }
const uint32_t* orc_expx_freqs_of(const orc_expx* f) { return f->freqs; }
const uint64_t* orc_expx_counts_of(const orc_expx* f) { return f->counts; }
const uint32_t* orc_expx_states(const orc_expx* f) { return f->states; }
const uint32_t* orc_expx_offsets(const orc_expx* f) { return f->offsets; }
uint16_t* orc_expx_payload_mut(orc_expx* f) { return f->payload; }
const uint32_t* orc_expx_rec_off(const orc_expx* f) { return f->rec_off; }
const uint32_t* orc_expx_records(const orc_expx* f) { return f->records; }
const uint8_t* orc_expx_sm(const orc_expx* f) { return f->sm; }
