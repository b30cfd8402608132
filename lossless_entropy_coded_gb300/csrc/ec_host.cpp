/*
 * ec_host.cpp -- host side of the library: the two encoders, the device blob, and
 * the bookkeeping entry points (ec_stats, ec_code_lengths, ec_free, ec_strerror).
 *
 * Huffman-exponent codec (DFloat11, "70% Size, 100% Accuracy", section
 * "Dynamic-Length Float" and Fig. 3): the exponent byte of every BF16 weight is
 * Huffman coded, one code per matrix; sign and mantissa stay one raw byte.
 * Codeword lengths come from Huffman's merge rule, or from package-merge when the
 * Huffman tree is deeper than the length limit; codewords are canonical.
 *
 * rANS codec (EntroPack section 3.6 / appendix C.3): 4-bit codes in independent
 * tiles decoded by one warp, 32 interleaved lanes, 32-bit states in [2^16, 2^32),
 * 16-bit renormalisation words.
 *
 * Sizes are computed with checked 64-bit arithmetic before any allocation
 * (loading-time rule from "M8.9 Quantized Artifacts and Runtime Integration",
 * section "Parse Before Allocation").
 */
#include <cuda_runtime.h>

#include <algorithm>
#include <array>
#include <atomic>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <queue>
#include <thread>
#include <vector>

#include "ec_internal.h"

static_assert(sizeof(ec_blob_header) == 256, "blob header must be 256 bytes");

namespace {

/* ------------------------------------------------------------------ utilities */
bool mul_ok(int64_t a, int64_t b, int64_t* r) {
    if (a < 0 || b < 0) return false;
    if (a != 0 && b > INT64_MAX / a) return false;
    *r = a * b;
    return true;
}
bool add_ok(int64_t a, int64_t b, int64_t* r) {
    if (a < 0 || b < 0 || a > INT64_MAX - b) return false;
    *r = a + b;
    return true;
}
int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }

/* Values at padded positions [base, base + n) of a row-major [rows, K] matrix laid
 * out with rows of KP >= K entries (the tail of each row reads as zero). */
template <class T>
void gather_padded(const T* src, int64_t K, int64_t KP, int64_t base, int64_t n, T* out) {
    int64_t r = base / KP, c = base - r * KP;
    for (int64_t q = 0; q < n;) {
        const int64_t run = std::min(n - q, KP - c);
        const T* row = src + r * K;
        for (int64_t k = 0; k < run; ++k) out[q + k] = (c + k < K) ? row[c + k] : T(0);
        q += run;
        c = 0;
        ++r;
    }
}

int host_threads() {
    unsigned n = std::thread::hardware_concurrency();
    if (n == 0) n = 4;
    return (int)std::min(n, 64u);
}

/* Run fn(lo, hi) over [0, n) split across threads. */
template <class F>
void parallel_for(int64_t n, F fn, int64_t min_chunk = 1) {
    int nt = host_threads();
    if (n / std::max<int64_t>(min_chunk, 1) < nt) nt = (int)std::max<int64_t>(1, n / std::max<int64_t>(min_chunk, 1));
    if (nt <= 1) {
        fn((int64_t)0, n);
        return;
    }
    std::vector<std::thread> th;
    th.reserve(nt);
    for (int t = 0; t < nt; ++t) th.emplace_back([=] { fn(n * t / nt, n * (t + 1) / nt); });
    for (auto& x : th) x.join();
}

/* --------------------------------------------------------- Huffman code lengths */

/* Huffman's merge rule with a priority queue; ties go to the node whose subtree
 * holds the smallest symbol.  Returns the number of present symbols. */
int huffman_lengths(const uint64_t counts[256], uint8_t len[256]) {
    struct Node {
        uint64_t w;
        int minsym, id;
    };
    auto later = [](const Node& a, const Node& b) { return a.w != b.w ? a.w > b.w : a.minsym > b.minsym; };
    std::priority_queue<Node, std::vector<Node>, decltype(later)> pq(later);
    std::vector<int> parent;
    std::vector<int> leaf(256, -1);
    for (int s = 0; s < 256; ++s) {
        if (!counts[s]) continue;
        leaf[s] = (int)parent.size();
        pq.push({counts[s], s, (int)parent.size()});
        parent.push_back(-1);
    }
    std::memset(len, 0, 256);
    const int n = (int)parent.size();
    if (n == 1) {
        for (int s = 0; s < 256; ++s)
            if (leaf[s] >= 0) len[s] = 1;
    }
    if (n <= 1) return n;
    while (pq.size() > 1) {
        Node a = pq.top();
        pq.pop();
        Node b = pq.top();
        pq.pop();
        const int id = (int)parent.size();
        parent.push_back(-1);
        parent[a.id] = parent[b.id] = id;
        pq.push({a.w + b.w, std::min(a.minsym, b.minsym), id});
    }
    for (int s = 0; s < 256; ++s) {
        if (leaf[s] < 0) continue;
        int d = 0;
        for (int v = leaf[s]; parent[v] >= 0; v = parent[v]) ++d;
        len[s] = (uint8_t)d;
    }
    return n;
}

/* Optimal code with lengths <= L: package-merge over L denominations.  Leaves are
 * ordered by (count, symbol); a package is the sum of two adjacent items of the
 * finer list; equal weights put the leaf first.  The coarsest list keeps 2(n-1)
 * items and a symbol's length is how often its leaf is inside them (tracked as a
 * per-item vector of leaf multiplicities, accumulated level by level). */
bool package_merge_lengths(const uint64_t counts[256], int L, uint8_t len[256]) {
    std::vector<int> sym;
    for (int s = 0; s < 256; ++s)
        if (counts[s]) sym.push_back(s);
    std::memset(len, 0, 256);
    const int n = (int)sym.size();
    if (n <= 1) {
        if (n == 1) len[sym[0]] = 1;
        return true;
    }
    if (L < 1 || L > 30 || (int64_t(1) << L) < n) return false;
    std::stable_sort(sym.begin(), sym.end(), [&](int a, int b) { return counts[a] < counts[b]; });
    /* An item is described by how many times each leaf (by rank) occurs in it. */
    struct Item {
        uint64_t w;
        std::vector<uint8_t> mult;
    };
    std::vector<Item> cur;
    for (int i = 0; i < n; ++i) {
        Item it{counts[sym[i]], std::vector<uint8_t>(n, 0)};
        it.mult[i] = 1;
        cur.push_back(std::move(it));
    }
    for (int level = 1; level < L; ++level) {
        std::vector<Item> next;
        next.reserve(2 * n);
        size_t li = 0, pi = 0;
        const size_t np = cur.size() / 2;
        while (li < (size_t)n || pi < np) {
            uint64_t pw = pi < np ? cur[2 * pi].w + cur[2 * pi + 1].w : 0;
            if (li < (size_t)n && (pi >= np || counts[sym[li]] <= pw)) {
                Item it{counts[sym[li]], std::vector<uint8_t>(n, 0)};
                it.mult[li] = 1;
                next.push_back(std::move(it));
                ++li;
            } else {
                Item it{pw, cur[2 * pi].mult};
                for (int k = 0; k < n; ++k) it.mult[k] = (uint8_t)(it.mult[k] + cur[2 * pi + 1].mult[k]);
                next.push_back(std::move(it));
                ++pi;
            }
        }
        cur.swap(next);
    }
    std::vector<int> total(n, 0);
    for (int i = 0; i < 2 * (n - 1); ++i)
        for (int k = 0; k < n; ++k) total[k] += cur[i].mult[k];
    for (int k = 0; k < n; ++k) len[sym[k]] = (uint8_t)total[k];
    return true;
}

/* Canonical codewords: ascending (length, symbol), consecutive values. */
void canonical(const uint8_t len[256], uint32_t code[256]) {
    std::vector<int> order;
    for (int s = 0; s < 256; ++s)
        if (len[s]) order.push_back(s);
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return len[a] < len[b]; });
    std::memset(code, 0, 256 * sizeof(uint32_t));
    uint32_t c = 0;
    for (size_t i = 0; i < order.size(); ++i) {
        if (i) c = (c + 1) << (len[order[i]] - len[order[i - 1]]);
        code[order[i]] = c;
    }
}

/* The codeword of length l with canonical value c, in stream order: its first
 * (most significant) bit becomes bit 0. */
uint32_t stream_bits(uint32_t c, int l) {
    uint32_t r = 0;
    for (int i = 0; i < l; ++i) r |= ((c >> (l - 1 - i)) & 1u) << i;
    return r;
}

/* Decode tables of the LSB-first stream (layout in ec_format.h).  one[w] names the
 * codeword that a 12-bit window w starts with: exponent << 7 | length << 16 for a
 * codeword that ends inside the window, EC_ENT_PTR for the 12-bit prefix of a
 * longer one, EC_ENT_BAD where nothing matches (corrupt data, or the unused half of
 * a one-symbol code's space). */
struct HuffTables {
    std::vector<uint32_t> pair; /* 2^EC_L1_BITS entries */
    std::vector<uint32_t> sub;  /* hierarchical sub-tables, 256 entries each */
};

HuffTables build_huff_tables(const uint8_t len[256], const uint32_t code[256], bool hierarchical) {
    const uint32_t W = EC_L1_BITS, mask = (1u << W) - 1;
    std::vector<uint32_t> one(1u << W, EC_ENT_BAD);
    HuffTables t;
    /* level-2 sub-table of each 12-bit prefix of a longer codeword, level-3 of each
     * 20-bit prefix of a codeword longer than 20 bits (codewords are at most 24) */
    std::vector<int> l2(1u << W, -1);
    std::vector<std::pair<uint32_t, int>> l3; /* (20-bit prefix, sub-table) */
    auto new_sub = [&]() {
        t.sub.resize(t.sub.size() + 256, EC_ENT_BAD);
        return (int)(t.sub.size() / 256 - 1);
    };
    for (int s = 0; s < 256; ++s) {
        const int l = len[s];
        if (!l) continue;
        const uint32_t bits = stream_bits(code[s], l), sym = ((uint32_t)s << 7) | ((uint32_t)l << 16);
        if (l <= (int)W) {
            for (uint32_t hi = 0; hi < (1u << (W - l)); ++hi) one[bits | (hi << l)] = sym;
            continue;
        }
        const uint32_t p12 = bits & mask;
        one[p12] = EC_ENT_PTR;
        if (!hierarchical) continue;
        if (l2[p12] < 0) l2[p12] = new_sub();
        const int t2 = l2[p12];
        const int rem = l - (int)W;
        if (rem <= 8) {
            for (uint32_t hi = 0; hi < (1u << (8 - rem)); ++hi) t.sub[256 * t2 + ((bits >> W) | (hi << rem))] = sym;
            continue;
        }
        const uint32_t p20 = bits & 0xFFFFFu, i2 = (bits >> W) & 0xFFu;
        int t3 = -1;
        for (auto& q : l3)
            if (q.first == p20) t3 = q.second;
        if (t3 < 0) {
            t3 = new_sub();
            l3.push_back({p20, t3});
            t.sub[256 * t2 + i2] = EC_ENT_PTR | (uint32_t)t3 | (20u << 16);
        }
        const int rem3 = l - 20;
        for (uint32_t hi = 0; hi < (1u << (8 - rem3)); ++hi) t.sub[256 * t3 + ((bits >> 20) | (hi << rem3))] = sym;
    }
    /* pair entries: the first codeword, and the second when it ends inside the window
     * too (the window shifted right by the first length names it; it counts only if
     * its length fits the bits that remain) */
    t.pair.assign(EC_PAIR_WORDS, 0);
    for (uint32_t w = 0; w <= mask; ++w) {
        const uint32_t a = one[w];
        if (a & EC_ENT_BAD) {
            t.pair[w] = EC_PAIR_OPEN;
            continue;
        }
        if (a & EC_ENT_PTR) { /* first codeword longer than the window: its sub-table */
            t.pair[w] = EC_PAIR_OPEN | (hierarchical ? ((uint32_t)l2[w] << 7) : 0u);
            continue;
        }
        const uint32_t l0 = (a >> 16) & 31, e0 = (a & 0xFFFFu) >> 7;
        uint32_t ent = (e0 << 7) | (l0 << EC_PAIR_FIRST_SHIFT);
        const uint32_t b = one[w >> l0];
        const uint32_t l1 = (b >> 16) & 31;
        if (!(b & (EC_ENT_PTR | EC_ENT_BAD)) && l0 + l1 <= W)
            ent |= (((b & 0xFFFFu) >> 7) << 23) | (l0 + l1);
        else
            ent |= EC_PAIR_OPEN | l0;
        t.pair[w] = ent;
    }
    return t;
}

/* Window records: the pairs (2m, 2m + 1) of one lane whose codewords do not both fit
 * the decoder's window get the shortest-coded exponent `fill` in place of one
 * exponent (the second when the first leaves room for fill's codeword, else the
 * first, and then the second too if it still does not fit).  e[] holds the lane's
 * exponents in symbol order and is rewritten; each substitution is reported with
 * rec(symbol index, true exponent).  Needs 2 len[fill] <= 12. */
template <class Rec>
void fit_pairs(uint8_t* e, int64_t S, const uint8_t len[256], int fill, Rec&& rec) {
    const int W = EC_L1_BITS, lf = len[fill];
    for (int64_t i = 0; i + 1 < S; i += 2) {
        const int la = len[e[i]], lb = len[e[i + 1]];
        if (la + lb <= W) continue;
        if (la + lf <= W) {
            rec(i + 1, e[i + 1]);
            e[i + 1] = (uint8_t)fill;
            continue;
        }
        rec(i, e[i]);
        e[i] = (uint8_t)fill;
        if (lf + lb > W) {
            rec(i + 1, e[i + 1]);
            e[i + 1] = (uint8_t)fill;
        }
    }
}

/* ------------------------------------------------------------ rANS frequencies */

/* f_s = max(1, floor(M c_s / n)) for present s; while the sum is short add one to
 * the present symbol with the largest remainder M c_s - f_s n, while it is over
 * take one from the present symbol with f_s > 1 and the smallest remainder (ties
 * to the lower symbol in both cases). */
bool rans_normalise(const uint64_t* counts, int nsym, int prob_bits, uint32_t* f) {
    const int64_t M = int64_t(1) << prob_bits;
    unsigned __int128 n = 0;
    int present = 0;
    for (int s = 0; s < nsym; ++s) {
        n += counts[s];
        present += counts[s] != 0;
    }
    std::memset(f, 0, (size_t)nsym * sizeof(uint32_t));
    if (n == 0) return true;
    if (present > M) return false;
    std::vector<__int128> rem((size_t)nsym, 0);
    int64_t sum = 0;
    for (int s = 0; s < nsym; ++s) {
        if (!counts[s]) continue;
        int64_t v = (int64_t)((unsigned __int128)M * counts[s] / n);
        v = std::max<int64_t>(v, 1);
        f[s] = (uint32_t)v;
        rem[s] = (__int128)M * counts[s] - (__int128)v * (__int128)n;
        sum += v;
    }
    for (; sum < M; ++sum) {
        int b = -1;
        for (int s = 0; s < nsym; ++s)
            if (counts[s] && (b < 0 || rem[s] > rem[b])) b = s;
        f[b]++;
        rem[b] -= (__int128)n;
    }
    for (; sum > M; --sum) {
        int b = -1;
        for (int s = 0; s < nsym; ++s)
            if (counts[s] && f[s] > 1 && (b < 0 || rem[s] < rem[b])) b = s;
        if (b < 0) return false;
        f[b]--;
        rem[b] += (__int128)n;
    }
    return true;
}

/* Table size for prob_bits = 0, MINE section 4.2 ("Launch"): candidate sizes 2^b,
 * b = 9..12, in increasing order, each scored by the cross-entropy lower bound of
 * the stored size, n * H(P, Q_b) bits of payload plus the table's 2^b 32-bit
 * entries; the scan stops once a score exceeds the best so far by more than 1%,
 * and the best is taken.  Returns 0 when no candidate can hold the alphabet. */
int rans_table_bits(const uint64_t* counts, int nsym) {
    int best_b = 0;
    double best = 0;
    std::vector<uint32_t> f(nsym);
    for (int b = 9; b <= 12; ++b) {
        if (!rans_normalise(counts, nsym, b, f.data())) continue;
        double bits = 32.0 * (double)(1u << b);
        for (int s = 0; s < nsym; ++s)
            if (counts[s]) bits -= (double)counts[s] * std::log2((double)f[s] / (double)(1u << b));
        if (best_b && bits > 1.01 * best) break;
        if (!best_b || bits < best) {
            best = bits;
            best_b = b;
        }
    }
    return best_b;
}

double entropy_bits(const uint64_t* c, int n) {
    double tot = 0, h = 0;
    for (int i = 0; i < n; ++i) tot += (double)c[i];
    if (tot <= 0) return 0;
    for (int i = 0; i < n; ++i)
        if (c[i]) {
            const double p = (double)c[i] / tot;
            h -= p * std::log2(p);
        }
    return h;
}

/* ------------------------------------------------------------------ device blob */
int upload(ec_matrix* m, const std::vector<uint8_t>& blob, int device) {
    if (device < 0) { /* host-only matrix: inspection and serialisation, no kernels */
        m->h_blob = (uint8_t*)std::malloc(std::max<size_t>(blob.size(), 1));
        if (!m->h_blob) return EC_ERR_OOM;
        std::memcpy(m->h_blob, blob.data(), blob.size());
        return EC_OK;
    }
    int prev = 0;
    if (cudaGetDevice(&prev) != cudaSuccess) return EC_ERR_CUDA;
    if (cudaSetDevice(device) != cudaSuccess) return EC_ERR_INVALID_ARG;
    void* p = nullptr;
    cudaError_t e = cudaMalloc(&p, std::max<size_t>(blob.size(), 256));
    if (e != cudaSuccess) {
        cudaGetLastError();
        cudaSetDevice(prev);
        return e == cudaErrorMemoryAllocation ? EC_ERR_OOM : EC_ERR_CUDA;
    }
    e = cudaMemcpy(p, blob.data(), blob.size(), cudaMemcpyHostToDevice);
    cudaSetDevice(prev);
    if (e != cudaSuccess) {
        cudaFree(p);
        return EC_ERR_CUDA;
    }
    m->d_blob = (uint8_t*)p;
    return EC_OK;
}

ec_matrix* new_matrix() {
    ec_matrix* m = new (std::nothrow) ec_matrix;
    if (m) std::memset((void*)m, 0, sizeof(ec_matrix));
    return m;
}

/* Encoder body under a try block: std::bad_alloc becomes EC_ERR_OOM. */
template <class F>
int guarded(F fn) {
    try {
        return fn();
    } catch (const std::bad_alloc&) {
        return EC_ERR_OOM;
    } catch (...) {
        return EC_ERR_INVALID_ARG;
    }
}

}  // namespace

/* ============================================================ Huffman encoder */
extern "C" int ec_encode_bf16(const uint16_t* w, int64_t n_rows, int64_t k_cols, const ec_huff_params* params,
                              int device, ec_matrix** out) {
    if (!out) return EC_ERR_INVALID_ARG;
    *out = nullptr;
    if (n_rows < 0 || k_cols < 0) return EC_ERR_SHAPE;
    const int max_len = params ? params->max_code_len : EC_DEFAULT_MAX_CODE_LEN;
    int steps = params ? params->tile_steps : 0;
    const int hier_req = params ? params->hierarchical : 0;
    if (max_len < 1 || max_len > EC_MAX_CODE_LEN) return EC_ERR_INVALID_ARG;
    if (steps < 0 || steps > EC_HUFF_MAX_STEPS || steps % 16) return EC_ERR_INVALID_ARG;
    if (hier_req != 0 && hier_req != 1) return EC_ERR_INVALID_ARG;
    int64_t nk = 0, k_pad = round_up(k_cols, EC_HUFF_ROW_ALIGN), n_pad = 0, tmp = 0;
    if (k_cols > INT64_MAX - EC_HUFF_ROW_ALIGN) return EC_ERR_OVERFLOW;
    if (!mul_ok(n_rows, k_cols, &nk) || !mul_ok(n_rows, k_pad, &n_pad) || !mul_ok(n_pad, 4, &tmp))
        return EC_ERR_OVERFLOW;
    if (steps == 0) { /* automatic: at least 1024 tiles where the matrix allows it, inside rows */
        steps = n_pad >= (int64_t)1024 * 32 * 128 ? 128 : n_pad >= (int64_t)1024 * 32 * 64 ? 64 : 32;
        while ((k_pad / 32) % steps) steps -= 16; /* k_pad / 32 is a multiple of 16 */
    }
    if (nk > 0 && !w) return EC_ERR_INVALID_ARG;

    return guarded([&]() -> int {
        const int64_t T = 32 * (int64_t)steps;
        const int64_t n_tiles = (n_pad + T - 1) / T;
        const int64_t K = k_cols, KP = k_pad;

        /* exponent histogram over the padded layout */
        const int nth = host_threads();
        std::vector<std::vector<uint64_t>> part(nth, std::vector<uint64_t>(256, 0));
        std::atomic<int> slot{0};
        parallel_for(
            n_rows,
            [&](int64_t lo, int64_t hi) {
                std::vector<uint64_t>& h = part[slot++ % nth];
                for (int64_t r = lo; r < hi; ++r) {
                    const uint16_t* row = w + r * K;
                    for (int64_t c = 0; c < K; ++c) h[(row[c] >> 7) & 0xFF]++;
                }
            },
            16);
        ec_matrix* m = new_matrix();
        if (!m) return EC_ERR_OOM;
        for (auto& h : part)
            for (int s = 0; s < 256; ++s) m->counts[s] += h[s];
        m->counts[0] += (uint64_t)(n_rows * (KP - K));

        if (huffman_lengths(m->counts, m->lengths) > 1) {
            int longest = *std::max_element(m->lengths, m->lengths + 256);
            if (longest > max_len && !package_merge_lengths(m->counts, max_len, m->lengths)) {
                delete m;
                return EC_ERR_INVALID_ARG;
            }
        }
        uint32_t code[256];
        canonical(m->lengths, code);
        /* the exponent with the shortest codeword fills pairs that overflow the window;
         * window records need two of its codewords to fit the window */
        int fill = -1;
        for (int s = 0; s < 256; ++s)
            if (m->lengths[s] && (fill < 0 || m->lengths[s] < m->lengths[fill])) fill = s;
        /* records pay when pairs rarely overflow: under independent exponents the share
         * of pairs with l(a) + l(b) > 12 must stay within 2 % (LLM weights: about 0.6 %) */
        double over = 0.0, tot = 0.0;
        for (int s = 0; s < 256; ++s) tot += (double)m->counts[s];
        for (int a = 0; a < 256 && tot > 0; ++a)
            for (int b = 0; b < 256; ++b)
                if (m->counts[a] && m->counts[b] && m->lengths[a] + m->lengths[b] > EC_L1_BITS)
                    over += (double)m->counts[a] / tot * ((double)m->counts[b] / tot);
        const bool records = !hier_req && (fill < 0 || (2 * m->lengths[fill] <= EC_L1_BITS && over <= 0.02));
        const HuffTables tabs = build_huff_tables(m->lengths, code, !records);
        if (tabs.sub.size() / 256 > 512) { /* sub-table indices have 9 bits */
            delete m;
            return EC_ERR_UNSUPPORTED;
        }
        std::vector<uint32_t> table = tabs.pair;
        table.insert(table.end(), tabs.sub.begin(), tabs.sub.end());

        /* A lane's exponents in symbol order (lane l owns tile positions 256 (i / 8) +
         * 8 l + i % 8), after window-record substitution; recs gets the records
         * (position in the tile | sign and mantissa << 13 | true exponent << 21). */
        auto lane_exponents = [&](const uint16_t* v, int64_t S, int l, uint8_t* e, std::vector<uint32_t>* recs) {
            for (int64_t i = 0; i < S; ++i) e[i] = (uint8_t)((v[256 * (i >> 3) + 8 * l + (i & 7)] >> 7) & 0xFF);
            if (records)
                fit_pairs(e, S, m->lengths, fill, [&](int64_t i, int true_e) {
                    if (recs) {
                        const uint32_t q = (uint32_t)(256 * (i >> 3) + 8 * l + (i & 7)), wq = v[q];
                        const uint32_t sm = ((wq >> 8) & 0x80u) | (wq & 0x7Fu);
                        recs->push_back(q | (sm << EC_HREC_SM_SHIFT) | ((uint32_t)true_e << EC_HREC_EXP_SHIFT));
                    }
                });
        };

        /* pass 1: per-tile record sizes and window records */
        std::vector<int64_t> rec_bytes(n_tiles + 1, 0), code_bytes(n_tiles, 0), n_rec(n_tiles, 0), bits_t(n_tiles, 0),
            area_bytes(n_tiles, 0);
        parallel_for(n_tiles, [&](int64_t lo, int64_t hi) {
            std::vector<uint16_t> v(T);
            std::vector<uint8_t> e(T / 32);
            std::vector<uint32_t> recs;
            for (int64_t t = lo; t < hi; ++t) {
                const int64_t base = t * T, n_t = std::min(T, n_pad - base), S = n_t / 32;
                gather_padded(w, K, KP, base, n_t, v.data());
                recs.clear();
                int64_t bytes = 0, bits_all = 0;
                for (int l = 0; l < 32; ++l) {
                    lane_exponents(v.data(), S, l, e.data(), &recs);
                    int64_t bits = 0;
                    for (int64_t i = 0; i < S; ++i) bits += m->lengths[e[i]];
                    bytes += (bits + 7) / 8;
                    bits_all += bits;
                }
                /* the tile's window records follow its code area */
                n_rec[t] = (int64_t)recs.size();
                area_bytes[t] = round_up(bytes + 8, 16);
                code_bytes[t] = area_bytes[t] + round_up(4 * n_rec[t], 16);
                rec_bytes[t] = 64 + EC_RAW_BYTES(n_t / 32) + code_bytes[t];
                bits_t[t] = bits_all;
            }
        });
        std::vector<uint32_t> tile_off(n_tiles + 1, 0);
        int64_t total = 0, max_code = 0, max_area = 0, payload = 0, n_records = 0;
        for (int64_t t = 0; t < n_tiles; ++t) {
            tile_off[t] = (uint32_t)(total / 16);
            if (!add_ok(total, rec_bytes[t], &total)) {
                delete m;
                return EC_ERR_OVERFLOW;
            }
            max_code = std::max(max_code, code_bytes[t]);
            max_area = std::max(max_area, area_bytes[t]);
            payload += bits_t[t];
            n_records += n_rec[t];
        }
        if (total / 16 > (int64_t)UINT32_MAX) {
            delete m;
            return EC_ERR_OVERFLOW;
        }
        tile_off[n_tiles] = (uint32_t)(total / 16);

        ec_blob_header h{};
        h.magic = EC_BLOB_MAGIC;
        h.version = EC_BLOB_VERSION;
        h.kind = EC_KIND_HUFFMAN_BF16;
        h.steps = steps;
        h.n_rows = n_rows;
        h.k_cols = k_cols;
        h.k_pad = KP;
        h.n_tiles = n_tiles;
        h.table_off = sizeof(ec_blob_header);
        h.table_words = (int64_t)table.size();
        h.scales_off = 0;
        h.huff_flags = records ? EC_HUFF_WINDOW_REC : 0;
        h.huff_fill = records && fill >= 0 ? fill : 0;
        h.huff_sub_tables = (int32_t)(tabs.sub.size() / 256);
        h.tile_off_off = round_up(h.table_off + 4 * h.table_words, 16);
        h.n_escapes = n_records;
        h.records_off = round_up(h.tile_off_off + 4 * (n_tiles + 1), 16);
        h.blob_bytes = h.records_off + total;
        h.max_code_bytes = (int32_t)max_code;
        h.max_code_area = (int32_t)max_area;
        h.max_len = *std::max_element(m->lengths, m->lengths + 256);
        {   /* staging size for the tensor-core kernel: a window of rows (tiles inside rows) */
            h.window_code_bytes = 0;
            if (KP % T == 0 && n_tiles > 0) {
                const int64_t R = KP / T;
                int64_t best = 0;
                for (int64_t tc = 0; tc < R; ++tc) {
                    int64_t sum = 0;
                    for (int64_t r = 0; r < n_rows; ++r) {
                        sum += 64 + code_bytes[r * R + tc];
                        if (r >= EC_MMA_WINDOW_ROWS) sum -= 64 + code_bytes[(r - EC_MMA_WINDOW_ROWS) * R + tc];
                        best = std::max(best, sum);
                    }
                }
                h.window_code_bytes = (int32_t)std::min<int64_t>(best, INT32_MAX);
            }
        }

        std::vector<uint8_t> blob((size_t)h.blob_bytes, 0);
        std::memcpy(blob.data(), &h, sizeof h);
        std::memcpy(blob.data() + h.table_off, table.data(), 4 * table.size());
        std::memcpy(blob.data() + h.tile_off_off, tile_off.data(), 4 * tile_off.size());

        /* pass 2: records */
        parallel_for(n_tiles, [&](int64_t lo, int64_t hi) {
            std::vector<uint16_t> v(T);
            std::vector<uint8_t> e(T / 32);
            std::vector<uint32_t> recs;
            for (int64_t t = lo; t < hi; ++t) {
                uint8_t* rec = blob.data() + h.records_off + (int64_t)tile_off[t] * 16;
                const int64_t base = t * T, n_t = std::min(T, n_pad - base), S = n_t / 32;
                gather_padded(w, K, KP, base, n_t, v.data());
                uint16_t* start = (uint16_t*)rec;
                uint8_t* raw = rec + 64;
                uint32_t* area = (uint32_t*)(rec + 64 + EC_RAW_BYTES(S));
                uint32_t* recs_at = area + area_bytes[t] / 4; /* the records follow the code area */
                /* sign / mantissa bytes: lane l, symbol i; in each group of four symbols
                 * the sign and mantissa bits of a pair sit where a BF16 pair keeps them,
                 * the second pair's rotated by 8 bits (ec_format.h) */
                for (int64_t q = 0; q < n_t; ++q) {
                    const int64_t l = (q >> 3) & 31, i = ((q >> 8) << 3) | (q & 7);
                    const uint8_t sg = (uint8_t)((v[q] >> 8) & 0x80), mt = (uint8_t)(v[q] & 0x7F);
                    uint8_t* g = raw + ((i >> 4) * 32 + l) * 16 + (i & 12); /* the group's four bytes */
                    switch (i & 3) {
                        case 0: g[0] |= mt; g[1] |= sg; break;
                        case 1: g[2] |= mt; g[3] |= sg; break;
                        case 2: g[1] |= mt; g[2] |= sg; break;
                        default: g[3] |= mt; g[0] |= sg; break;
                    }
                }
                recs.clear();
                int64_t bitpos = 0;
                for (int l = 0; l < 32; ++l) {
                    bitpos = round_up(bitpos, 8);
                    if (l) start[l] = (uint16_t)(bitpos / 8);
                    lane_exponents(v.data(), S, l, e.data(), &recs);
                    for (int64_t i = 0; i < S; ++i) {
                        const int L = m->lengths[e[i]];
                        const uint32_t c = stream_bits(code[e[i]], L);
                        const int64_t wi = bitpos >> 5;
                        const int o = (int)(bitpos & 31);
                        area[wi] |= c << o;
                        if (o + L > 32) area[wi + 1] |= c >> (32 - o);
                        bitpos += L;
                    }
                }
                /* lane 0 always starts at byte 0: its slot holds the record count */
                start[0] = (uint16_t)recs.size();
                std::sort(recs.begin(), recs.end(),
                          [](uint32_t x, uint32_t y) { return (x & EC_HREC_POS_MASK) < (y & EC_HREC_POS_MASK); });
                std::memcpy(recs_at, recs.data(), 4 * recs.size());
            }
        });

        m->kind = EC_KIND_HUFFMAN_BF16;
        m->device = device;
        m->hdr = h;
        m->payload_bits = payload;
        m->raw_bytes = n_pad;
        m->table_bytes = 4 * (int64_t)table.size();
        m->aux_bytes = h.blob_bytes - m->table_bytes - n_pad - (payload + 7) / 8;
        m->entropy = entropy_bits(m->counts, 256);
        int rc = upload(m, blob, device);
        if (rc != EC_OK) {
            delete m;
            return rc;
        }
        *out = m;
        return EC_OK;
    });
}

/* =============================================================== rANS encoder */
extern "C" int ec_encode_rans(const int8_t* codes, const uint16_t* scales, int64_t n_rows, int64_t k_cols,
                              const ec_rans_params* params, int device, ec_matrix** out) {
    if (!out) return EC_ERR_INVALID_ARG;
    *out = nullptr;
    if (n_rows < 0 || k_cols < 0) return EC_ERR_SHAPE;
    const int b_req = params ? params->prob_bits : 12; /* 0: chosen from the histogram */
    const int T = params ? params->tile_syms : 4096;
    const int group = params ? params->group : 128;
    const int k = params && params->codes_per_symbol ? params->codes_per_symbol : 1;
    const int values = params ? params->values : EC_RANS_VALUES_INT4;
    if (values != EC_RANS_VALUES_INT4 && values != EC_RANS_VALUES_FP4_E2M1) return EC_ERR_INVALID_ARG;
    if ((b_req != 0 && (b_req < 9 || b_req > 15)) || T < 32 || T % EC_RANS_ROW_ALIGN || T > 65536)
        return EC_ERR_INVALID_ARG;
    if (k != 1 && k != 2) return EC_ERR_INVALID_ARG;
    if (k == 2 && b_req > 12) return EC_ERR_INVALID_ARG; /* pair entries hold freq - 1 and the slot bias in 12 bits */
    if (group != 128) return EC_ERR_UNSUPPORTED;
    if (k_cols > INT64_MAX - EC_RANS_ROW_ALIGN) return EC_ERR_OVERFLOW;
    const int64_t KP = round_up(k_cols, EC_RANS_ROW_ALIGN), G = KP / 128;
    int64_t nk = 0, n_pad = 0, ns = 0, tmp = 0;
    if (!mul_ok(n_rows, k_cols, &nk) || !mul_ok(n_rows, KP, &n_pad) || !mul_ok(n_rows, G, &ns) ||
        !mul_ok(n_pad, 4, &tmp))
        return EC_ERR_OVERFLOW;
    if (nk > 0 && (!codes || !scales)) return EC_ERR_INVALID_ARG;

    return guarded([&]() -> int {
        const int64_t K = k_cols;
        /* FP4 E2M1 patterns 0..15 are coded as the 4-bit codes c - 8: the stream and
         * tables are the integer codec's, the header says how the decoder reads them */
        std::vector<int8_t> shifted;
        const int8_t* cv = codes;
        if (values == EC_RANS_VALUES_FP4_E2M1) {
            shifted.resize((size_t)nk);
            for (int64_t i = 0; i < nk; ++i) {
                if (codes[i] < 0 || codes[i] > 15) return EC_ERR_INVALID_ARG;
                shifted[(size_t)i] = (int8_t)(codes[i] - 8);
            }
            cv = shifted.data();
        }
        for (int64_t i = 0; i < nk; ++i)
            if (cv[i] < -8 || cv[i] > 7) return EC_ERR_INVALID_ARG;
        ec_matrix* m = new_matrix();
        if (!m) return EC_ERR_OOM;
        const int nsym = k == 1 ? 16 : 256;
        const int64_t n_tiles = (n_pad + T - 1) / T;
        /* symbol of lane l's symbol step j in a tile's padded codes v */
        auto symbol = [k](const int8_t* v, int64_t j, int l) {
            return k == 1 ? v[32 * j + l] + 8 : 16 * (v[64 * j + l] + 8) + (v[64 * j + 32 + l] + 8);
        };
        if (k == 1) {
            for (int64_t i = 0; i < nk; ++i) m->counts[cv[i] + 8]++;
            m->counts[8] += (uint64_t)(n_rows * (KP - K));
        } else { /* histogram of the pair symbols over the padded tile layout */
            std::vector<std::array<uint64_t, 256>> part(host_threads());
            for (auto& a : part) a.fill(0);
            std::atomic<int> slot{0};
            parallel_for(
                n_tiles,
                [&](int64_t lo, int64_t hi) {
                    auto& hcount = part[slot++ % part.size()];
                    std::vector<int8_t> v(T);
                    for (int64_t t = lo; t < hi; ++t) {
                        const int64_t base = t * T, n_t = std::min<int64_t>(T, n_pad - base), S = n_t / 32;
                        gather_padded(cv, K, KP, base, n_t, v.data());
                        for (int64_t j = 0; j < S / 2; ++j)
                            for (int l = 0; l < 32; ++l) hcount[symbol(v.data(), j, l)]++;
                    }
                }); /* at most one chunk per thread: one histogram each */
            for (auto& a : part)
                for (int s = 0; s < 256; ++s) m->counts[s] += a[s];
        }
        const int b = b_req ? b_req : rans_table_bits(m->counts, nsym);
        if (!b || !rans_normalise(m->counts, nsym, b, m->freqs)) {
            delete m;
            return EC_ERR_INVALID_ARG;
        }
        const uint32_t M = 1u << b;
        std::vector<uint32_t> cum(nsym, 0);
        for (int s = 0, c = 0; s < nsym; ++s) {
            cum[s] = (uint32_t)c;
            c += (int)m->freqs[s];
        }
        std::vector<uint32_t> table(M, 0);
        for (int s = 0; s < nsym; ++s)
            for (uint32_t q = 0; q < m->freqs[s]; ++q)
                table[cum[s] + q] = k == 1 ? (uint32_t)s | (q << 4) | (m->freqs[s] << 16)
                                           : (uint32_t)s | (q << 8) | ((m->freqs[s] - 1) << 20);

        std::vector<std::vector<uint16_t>> words(n_tiles);
        std::vector<std::array<uint32_t, 32>> states(n_tiles);
        const uint64_t unit = uint64_t(1) << (32 - b);
        parallel_for(n_tiles, [&](int64_t lo, int64_t hi) {
            std::vector<uint16_t> stack;
            std::vector<int8_t> v(T);
            for (int64_t t = lo; t < hi; ++t) {
                const int64_t base = t * T, n_t = std::min<int64_t>(T, n_pad - base), S = n_t / 32;
                gather_padded(cv, K, KP, base, n_t, v.data());
                uint64_t x[32];
                for (int l = 0; l < 32; ++l) x[l] = 1u << 16;
                stack.clear();
                for (int64_t j = S / k - 1; j >= 0; --j)
                    for (int l = 31; l >= 0; --l) {
                        const int s = symbol(v.data(), j, l);
                        const uint64_t f = m->freqs[s];
                        if (x[l] >= f * unit) {
                            stack.push_back((uint16_t)x[l]);
                            x[l] >>= 16;
                        }
                        x[l] = ((x[l] / f) << b) + x[l] % f + cum[s];
                    }
                for (int l = 0; l < 32; ++l) states[t][l] = (uint32_t)x[l];
                words[t].assign(stack.rbegin(), stack.rend());
            }
        });
        std::vector<uint32_t> tile_off(n_tiles + 1, 0);
        int64_t total = 0, max_words = 0, payload = 0;
        for (int64_t t = 0; t < n_tiles; ++t) {
            tile_off[t] = (uint32_t)(total / 16);
            total += 128 + round_up(2 * (int64_t)words[t].size(), 16);
            max_words = std::max<int64_t>(max_words, (int64_t)words[t].size());
            payload += 16 * (int64_t)words[t].size();
        }
        if (total / 16 > (int64_t)UINT32_MAX) {
            delete m;
            return EC_ERR_OVERFLOW;
        }
        tile_off[n_tiles] = (uint32_t)(total / 16);

        ec_blob_header h{};
        h.magic = EC_BLOB_MAGIC;
        h.version = EC_BLOB_VERSION;
        h.kind = EC_KIND_RANS_INT4;
        h.steps = T / 32;
        h.n_rows = n_rows;
        h.k_cols = k_cols;
        h.k_pad = KP;
        h.n_tiles = n_tiles;
        h.table_off = sizeof(ec_blob_header);
        h.table_words = M;
        h.scales_off = round_up(h.table_off + 4 * (int64_t)M, 16);
        h.tile_off_off = round_up(h.scales_off + 2 * ns, 16);
        h.records_off = round_up(h.tile_off_off + 4 * (n_tiles + 1), 16);
        h.blob_bytes = h.records_off + total;
        h.prob_bits = b;
        h.max_words = (int32_t)max_words;
        h.rans_tuple = k;
        h.rans_values = values;

        std::vector<uint8_t> blob((size_t)h.blob_bytes, 0);
        std::memcpy(blob.data(), &h, sizeof h);
        std::memcpy(blob.data() + h.table_off, table.data(), 4 * table.size());
        if (ns) std::memcpy(blob.data() + h.scales_off, scales, 2 * (size_t)ns);
        std::memcpy(blob.data() + h.tile_off_off, tile_off.data(), 4 * tile_off.size());
        parallel_for(n_tiles, [&](int64_t lo, int64_t hi) {
            for (int64_t t = lo; t < hi; ++t) {
                uint8_t* rec = blob.data() + h.records_off + (int64_t)tile_off[t] * 16;
                std::memcpy(rec, states[t].data(), 128);
                if (!words[t].empty()) std::memcpy(rec + 128, words[t].data(), 2 * words[t].size());
            }
        });
        m->kind = EC_KIND_RANS_INT4;
        m->device = device;
        m->hdr = h;
        m->payload_bits = payload;
        m->raw_bytes = 0;
        m->table_bytes = 4 * (int64_t)M + 2 * ns;
        m->aux_bytes = h.blob_bytes - m->table_bytes - payload / 8;
        m->entropy = entropy_bits(m->counts, nsym) / k; /* bits per code */
        int rc = upload(m, blob, device);
        if (rc != EC_OK) {
            delete m;
            return rc;
        }
        *out = m;
        return EC_OK;
    });
}

/* ============================================================ E8 lattice encoder */
namespace {
/* Fields of a doubled E8 point q[8] (EntroPack sections 3.2, 3.3; appendix A.3):
 * the coset c = q_1 mod 2, z_j = (q_j - c) / 2 (j = 1..7) offset by 16, and the
 * parity-reduced m = (z_8 - (z_1 + .. + z_7) mod 2) / 2 offset by 16.  False if q is
 * not in 2 E8 or a field leaves its alphabet. */
bool e8_point_fields(const int8_t* q, int* fld) {
    const int c = q[0] & 1;
    int z[8], sum = 0;
    for (int j = 0; j < 8; ++j) {
        if ((q[j] & 1) != c) return false;
        z[j] = (q[j] - c) / 2;
        sum += z[j];
    }
    if (sum & 1) return false; /* not in D8 */
    const int par = (sum - z[7]) & 1;
    const int m = (z[7] - par) / 2;
    fld[0] = c;
    for (int j = 0; j < 7; ++j) {
        if (z[j] < -16 || z[j] > 15) return false;
        fld[1 + j] = z[j] + 16;
    }
    if (m < -8 || m > 7) return false;
    fld[8] = m + 16;
    return true;
}
inline int e8_table_of(int f, int c) { return f == 0 ? 0 : 1 + 8 * c + (f - 1); }
}  // namespace

extern "C" int ec_encode_e8(const int8_t* q2, const float* row_scales, float scale, int64_t n_rows, int64_t k_cols,
                            const ec_e8_params* params, int device, ec_matrix** out) {
    if (!out) return EC_ERR_INVALID_ARG;
    *out = nullptr;
    if (n_rows < 0 || k_cols < 0 || k_cols % 8) return EC_ERR_SHAPE;
    const int b = params && params->prob_bits ? params->prob_bits : 11;
    const int TV = params && params->tile_vectors ? params->tile_vectors : 1024;
    if (b < 9 || b > 12 || TV < 32 || TV % 32 || TV > 1024) return EC_ERR_INVALID_ARG;
    if (!std::isfinite(scale)) return EC_ERR_INVALID_ARG;
    if (k_cols > INT64_MAX - EC_E8_ROW_ALIGN) return EC_ERR_OVERFLOW;
    const int64_t KP = round_up(k_cols, EC_E8_ROW_ALIGN), VPR = KP / 8;
    int64_t nk = 0, n_vec = 0, tmp = 0;
    if (!mul_ok(n_rows, k_cols, &nk) || !mul_ok(n_rows, VPR, &n_vec) || !mul_ok(n_vec, 9 * 2, &tmp))
        return EC_ERR_OVERFLOW;
    if (nk > 0 && (!q2 || !row_scales)) return EC_ERR_INVALID_ARG;

    return guarded([&]() -> int {
        const int64_t K = k_cols;
        /* fields of every vector of the padded layout (padding: the zero point) */
        std::vector<uint8_t> fields((size_t)n_vec * 9, 0);
        std::atomic<bool> bad{false};
        parallel_for(n_rows, [&](int64_t lo, int64_t hi) {
            int f[9];
            for (int64_t r = lo; r < hi && !bad; ++r)
                for (int64_t v = 0; v < VPR; ++v) {
                    uint8_t* dst = fields.data() + 9 * (r * VPR + v);
                    if (8 * v < K) {
                        if (!e8_point_fields(q2 + r * K + 8 * v, f)) {
                            bad = true;
                            break;
                        }
                        for (int i = 0; i < 9; ++i) dst[i] = (uint8_t)f[i];
                    } else {
                        dst[0] = 0;
                        for (int i = 1; i < 9; ++i) dst[i] = 16;
                    }
                }
        });
        if (bad) return EC_ERR_INVALID_ARG;
        for (int64_t r = 0; r < n_rows; ++r) /* the decoder's row factor fp32(s * r_i) must be finite */
            if (!std::isfinite(row_scales[r]) || !std::isfinite(scale * row_scales[r])) return EC_ERR_INVALID_ARG;
        ec_matrix* m = new_matrix();
        if (!m) return EC_ERR_OOM;
        uint64_t counts[EC_E8_TABLES][EC_E8_ALPHA] = {};
        for (int64_t v = 0; v < n_vec; ++v) {
            const uint8_t* fv = fields.data() + 9 * v;
            for (int f = 0; f < 9; ++f) counts[e8_table_of(f, fv[0])][fv[f]]++;
        }
        const uint32_t M = 1u << b;
        uint32_t freq[EC_E8_TABLES][EC_E8_ALPHA] = {}, cum[EC_E8_TABLES][EC_E8_ALPHA] = {};
        std::vector<uint8_t> slot_sym((size_t)EC_E8_TABLES * M, 0);
        double ideal_bits = 0;
        for (int t = 0; t < EC_E8_TABLES; ++t) {
            uint64_t n_t = 0;
            for (int s = 0; s < EC_E8_ALPHA; ++s) n_t += counts[t][s];
            if (!n_t) continue; /* a table no symbol uses (a coset that never occurs) */
            if (!rans_normalise(counts[t], EC_E8_ALPHA, b, freq[t])) {
                delete m;
                return EC_ERR_INVALID_ARG;
            }
            for (int s = 0, c = 0; s < EC_E8_ALPHA; ++s) {
                cum[t][s] = (uint32_t)c;
                for (uint32_t q = 0; q < freq[t][s]; ++q) slot_sym[(size_t)t * M + c + q] = (uint8_t)s;
                c += (int)freq[t][s];
                if (counts[t][s]) ideal_bits -= (double)counts[t][s] * std::log2((double)counts[t][s] / (double)n_t);
            }
        }
        /* tiles: vector j of lane l is tile vector 32 j + l; encoded last vector first,
         * fields 8 -> 0, lanes 31 -> 0, so the decoder reads in the opposite order */
        const int64_t n_tiles = (n_vec + TV - 1) / TV;
        std::vector<std::vector<uint16_t>> words(n_tiles);
        std::vector<std::array<uint32_t, 32>> states(n_tiles);
        const uint64_t unit = uint64_t(1) << (32 - b);
        parallel_for(n_tiles, [&](int64_t lo, int64_t hi) {
            std::vector<uint16_t> stack;
            for (int64_t t = lo; t < hi; ++t) {
                const int64_t base = t * TV, n_t = std::min<int64_t>(TV, n_vec - base);
                uint64_t x[32];
                for (int l = 0; l < 32; ++l) x[l] = 1u << 16;
                stack.clear();
                for (int64_t j = (n_t + 31) / 32 - 1; j >= 0; --j)
                    for (int f = 8; f >= 0; --f)
                        for (int l = 31; l >= 0; --l) {
                            if (32 * j + l >= n_t) continue;
                            const uint8_t* fv = fields.data() + 9 * (base + 32 * j + l);
                            const int tb = e8_table_of(f, fv[0]), s = fv[f];
                            const uint64_t fr = freq[tb][s];
                            while (x[l] >= fr * unit) {
                                stack.push_back((uint16_t)(x[l] & 0xFFFF));
                                x[l] >>= 16;
                            }
                            x[l] = (x[l] / fr << b) + (x[l] % fr) + cum[tb][s];
                        }
                for (int l = 0; l < 32; ++l) states[t][l] = (uint32_t)x[l];
                words[t].assign(stack.rbegin(), stack.rend());
            }
        });
        std::vector<uint32_t> tile_off(n_tiles + 1, 0);
        int64_t total = 0, max_words = 0, payload = 0;
        for (int64_t t = 0; t < n_tiles; ++t) {
            tile_off[t] = (uint32_t)(total / 16);
            total += 128 + round_up(2 * (int64_t)words[t].size(), 16);
            max_words = std::max<int64_t>(max_words, (int64_t)words[t].size());
            payload += 16 * (int64_t)words[t].size();
        }
        if (total / 16 > (int64_t)UINT32_MAX) {
            delete m;
            return EC_ERR_OVERFLOW;
        }
        tile_off[n_tiles] = (uint32_t)(total / 16);

        const int64_t fc_words = EC_E8_TABLES * EC_E8_ALPHA, table_bytes = 4 * fc_words + (int64_t)EC_E8_TABLES * M;
        ec_blob_header h{};
        h.magic = EC_BLOB_MAGIC;
        h.version = EC_BLOB_VERSION;
        h.kind = EC_KIND_E8;
        h.steps = TV / 32;
        h.n_rows = n_rows;
        h.k_cols = k_cols;
        h.k_pad = KP;
        h.n_tiles = n_tiles;
        h.table_off = sizeof(ec_blob_header);
        h.table_words = table_bytes / 4;
        h.scales_off = round_up(h.table_off + table_bytes, 16);
        h.tile_off_off = round_up(h.scales_off + 4 * n_rows, 16);
        h.records_off = round_up(h.tile_off_off + 4 * (n_tiles + 1), 16);
        h.blob_bytes = h.records_off + total;
        h.prob_bits = b;
        h.max_words = (int32_t)max_words;
        std::memcpy(&h.e8_scale_bits, &scale, 4);

        std::vector<uint8_t> blob((size_t)h.blob_bytes, 0);
        std::memcpy(blob.data(), &h, sizeof h);
        uint32_t* fc = (uint32_t*)(blob.data() + h.table_off);
        for (int t = 0; t < EC_E8_TABLES; ++t)
            for (int s = 0; s < EC_E8_ALPHA; ++s) fc[t * EC_E8_ALPHA + s] = freq[t][s] | (cum[t][s] << 16);
        std::memcpy(blob.data() + h.table_off + 4 * fc_words, slot_sym.data(), slot_sym.size());
        if (n_rows) std::memcpy(blob.data() + h.scales_off, row_scales, 4 * (size_t)n_rows);
        std::memcpy(blob.data() + h.tile_off_off, tile_off.data(), 4 * tile_off.size());
        parallel_for(n_tiles, [&](int64_t lo, int64_t hi) {
            for (int64_t t = lo; t < hi; ++t) {
                uint8_t* rec = blob.data() + h.records_off + (int64_t)tile_off[t] * 16;
                std::memcpy(rec, states[t].data(), 128);
                if (!words[t].empty()) std::memcpy(rec + 128, words[t].data(), 2 * words[t].size());
            }
        });
        m->kind = EC_KIND_E8;
        m->device = device;
        m->hdr = h;
        m->payload_bits = payload;
        m->raw_bytes = 0;
        m->table_bytes = table_bytes + 4 * n_rows;
        m->aux_bytes = h.blob_bytes - m->table_bytes - payload / 8;
        m->entropy = n_vec ? ideal_bits / (8.0 * (double)n_vec) : 0.0; /* ideal bits per weight, conditioned tables */
        int rc = upload(m, blob, device);
        if (rc != EC_OK) {
            delete m;
            return rc;
        }
        *out = m;
        return EC_OK;
    });
}

/* ============================================================ FP8 top-t encoder */
/* MINE section 4, "Escapes": the decoding table keeps the t most frequent codes, 0
 * always among them; any other weight is coded as 0 and its code goes to a sparse
 * correction stream of 32-bit records. */
namespace {
/* Value of an OCP FP8 E4M3 code: sign, exponent field e (bias 7), mantissa m; e = 0
 * holds the subnormals m/8 * 2^-6; S.1111.111 is NaN. */
float e4m3_value(int code) {
    const int s = code >> 7, e = (code >> 3) & 15, m = code & 7;
    if (e == 15 && m == 7) return std::nanf("");
    const float v = e == 0 ? std::ldexp((float)m / 8.0f, -6) : std::ldexp(1.0f + (float)m / 8.0f, e - 7);
    return s ? -v : v;
}
}  // namespace

extern "C" int ec_encode_fp8(const uint8_t* codes, const float* row_scales, int64_t n_rows, int64_t k_cols,
                             const ec_fp8_params* params, int device, ec_matrix** out) {
    if (!out) return EC_ERR_INVALID_ARG;
    *out = nullptr;
    if (n_rows < 0 || k_cols < 0) return EC_ERR_SHAPE;
    const int b = params && params->prob_bits ? params->prob_bits : 12;
    const int T = params && params->tile_syms ? params->tile_syms : 4096;
    const int t_req = params ? params->top_t : 0;
    if (b < 9 || b > 12 || T < EC_RANS_ROW_ALIGN || T % EC_RANS_ROW_ALIGN || T > 4096 || t_req < 0 || t_req > 256)
        return EC_ERR_INVALID_ARG;
    if (k_cols > INT64_MAX - EC_RANS_ROW_ALIGN) return EC_ERR_OVERFLOW;
    const int64_t KP = round_up(k_cols, EC_RANS_ROW_ALIGN);
    int64_t nk = 0, n_pad = 0, tmp = 0;
    if (!mul_ok(n_rows, k_cols, &nk) || !mul_ok(n_rows, KP, &n_pad) || !mul_ok(n_pad, 4, &tmp)) return EC_ERR_OVERFLOW;
    if (nk > 0 && (!codes || !row_scales)) return EC_ERR_INVALID_ARG;

    return guarded([&]() -> int {
        const int64_t K = k_cols;
        for (int64_t i = 0; i < nk; ++i)
            if ((codes[i] & 0x7F) == 0x7F) return EC_ERR_INVALID_ARG; /* NaN */
        for (int64_t r = 0; r < n_rows; ++r)
            if (!std::isfinite(row_scales[r])) return EC_ERR_INVALID_ARG;
        uint64_t hist[256] = {};
        for (int64_t i = 0; i < nk; ++i) hist[codes[i]]++;
        hist[0] += (uint64_t)(n_pad - nk); /* padding */
        /* the table: code 0, then the most frequent other present codes (ties to the
         * lower code) up to t, sorted by code; rank = symbol */
        const int t = t_req ? t_req : 256;
        bool kept[256] = {};
        kept[0] = true;
        for (int size = 1; size < t; ++size) {
            int best = -1;
            for (int c = 1; c < 256; ++c)
                if (!kept[c] && hist[c] && (best < 0 || hist[c] > hist[best])) best = c;
            if (best < 0) break;
            kept[best] = true;
        }
        int rank[256], tsize = 0;
        uint8_t table_codes[256] = {};
        for (int c = 0; c < 256; ++c) {
            rank[c] = kept[c] ? tsize : -1;
            if (kept[c]) table_codes[tsize++] = (uint8_t)c;
        }
        ec_matrix* m = new_matrix();
        if (!m) return EC_ERR_OOM;
        for (int c = 0; c < 256; ++c) m->counts[rank[c] >= 0 ? rank[c] : 0] += hist[c];
        if (!rans_normalise(m->counts, tsize, b, m->freqs)) {
            delete m;
            return EC_ERR_INVALID_ARG;
        }
        const uint32_t M = 1u << b;
        std::vector<uint32_t> cum(tsize, 0);
        for (int s = 0, c = 0; s < tsize; ++s) {
            cum[s] = (uint32_t)c;
            c += (int)m->freqs[s];
        }
        std::vector<uint32_t> table(M + EC_FP8_VALUE_WORDS, 0);
        for (int s = 0; s < tsize; ++s)
            for (uint32_t q = 0; q < m->freqs[s]; ++q)
                table[cum[s] + q] = (uint32_t)s | (q << 8) | ((m->freqs[s] - 1) << 20);
        for (int s = 0; s < tsize; ++s) {
            const float v = e4m3_value(table_codes[s]);
            std::memcpy(&table[M + s], &v, 4);
        }
        for (int c = 0; c < 256; ++c) {
            const float v = e4m3_value(c);
            std::memcpy(&table[M + 256 + c], &v, 4);
        }

        const int64_t n_tiles = (n_pad + T - 1) / T;
        std::vector<std::vector<uint16_t>> words(n_tiles);
        std::vector<std::vector<uint32_t>> recs(n_tiles);
        std::vector<std::array<uint32_t, 32>> states(n_tiles);
        const uint64_t unit = uint64_t(1) << (32 - b);
        parallel_for(n_tiles, [&](int64_t lo, int64_t hi) {
            std::vector<uint16_t> stack;
            std::vector<uint8_t> v(T);
            for (int64_t tt = lo; tt < hi; ++tt) {
                const int64_t base = tt * T, n_t = std::min<int64_t>(T, n_pad - base), S = n_t / 32;
                gather_padded(codes, K, KP, base, n_t, v.data());
                for (int64_t p = 0; p < n_t; ++p)
                    if (rank[v[p]] < 0) recs[tt].push_back((uint32_t)p | ((uint32_t)v[p] << 16));
                uint64_t x[32];
                for (int l = 0; l < 32; ++l) x[l] = 1u << 16;
                stack.clear();
                for (int64_t j = S - 1; j >= 0; --j)
                    for (int l = 31; l >= 0; --l) {
                        const int r = rank[v[32 * j + l]], s = r >= 0 ? r : 0;
                        const uint64_t f = m->freqs[s];
                        if (x[l] >= f * unit) {
                            stack.push_back((uint16_t)x[l]);
                            x[l] >>= 16;
                        }
                        x[l] = ((x[l] / f) << b) + x[l] % f + cum[s];
                    }
                for (int l = 0; l < 32; ++l) states[tt][l] = (uint32_t)x[l];
                words[tt].assign(stack.rbegin(), stack.rend());
            }
        });
        std::vector<uint32_t> tile_off(n_tiles + 1, 0), esc_off(n_tiles + 1, 0);
        int64_t total = 0, max_words = 0, payload = 0, n_esc = 0;
        for (int64_t tt = 0; tt < n_tiles; ++tt) {
            tile_off[tt] = (uint32_t)(total / 16);
            total += 128 + round_up(2 * (int64_t)words[tt].size(), 16);
            max_words = std::max<int64_t>(max_words, (int64_t)words[tt].size());
            payload += 16 * (int64_t)words[tt].size();
            esc_off[tt] = (uint32_t)n_esc;
            n_esc += (int64_t)recs[tt].size();
        }
        if (total / 16 > (int64_t)UINT32_MAX || n_esc > (int64_t)UINT32_MAX) {
            delete m;
            return EC_ERR_OVERFLOW;
        }
        tile_off[n_tiles] = (uint32_t)(total / 16);
        esc_off[n_tiles] = (uint32_t)n_esc;

        ec_blob_header h{};
        h.magic = EC_BLOB_MAGIC;
        h.version = EC_BLOB_VERSION;
        h.kind = EC_KIND_RANS_FP8;
        h.steps = T / 32;
        h.n_rows = n_rows;
        h.k_cols = k_cols;
        h.k_pad = KP;
        h.n_tiles = n_tiles;
        h.table_off = sizeof(ec_blob_header);
        h.table_words = (int64_t)M + EC_FP8_VALUE_WORDS;
        h.scales_off = round_up(h.table_off + 4 * h.table_words, 16);
        h.tile_off_off = round_up(h.scales_off + 4 * n_rows, 16);
        h.esc_off_off = round_up(h.tile_off_off + 4 * (n_tiles + 1), 16);
        h.esc_records_off = round_up(h.esc_off_off + 4 * (n_tiles + 1), 16);
        h.records_off = round_up(h.esc_records_off + 4 * n_esc, 16);
        h.blob_bytes = h.records_off + total;
        h.prob_bits = b;
        h.max_words = (int32_t)max_words;
        h.rans_tuple = 1;
        h.fp8_table_size = tsize;
        h.n_escapes = n_esc;

        std::vector<uint8_t> blob((size_t)h.blob_bytes, 0);
        std::memcpy(blob.data(), &h, sizeof h);
        std::memcpy(blob.data() + h.table_off, table.data(), 4 * table.size());
        if (n_rows) std::memcpy(blob.data() + h.scales_off, row_scales, 4 * (size_t)n_rows);
        std::memcpy(blob.data() + h.tile_off_off, tile_off.data(), 4 * tile_off.size());
        std::memcpy(blob.data() + h.esc_off_off, esc_off.data(), 4 * esc_off.size());
        parallel_for(n_tiles, [&](int64_t lo, int64_t hi) {
            for (int64_t tt = lo; tt < hi; ++tt) {
                uint8_t* rec = blob.data() + h.records_off + (int64_t)tile_off[tt] * 16;
                std::memcpy(rec, states[tt].data(), 128);
                if (!words[tt].empty()) std::memcpy(rec + 128, words[tt].data(), 2 * words[tt].size());
                if (!recs[tt].empty())
                    std::memcpy(blob.data() + h.esc_records_off + 4 * (int64_t)esc_off[tt], recs[tt].data(),
                                4 * recs[tt].size());
            }
        });
        m->kind = EC_KIND_RANS_FP8;
        m->device = device;
        m->hdr = h;
        m->payload_bits = payload + 32 * n_esc;
        m->raw_bytes = 0;
        m->table_bytes = 4 * h.table_words + 4 * n_rows;
        m->aux_bytes = h.blob_bytes - m->table_bytes - m->payload_bits / 8;
        m->entropy = entropy_bits(hist, 256); /* bits per code */
        int rc = upload(m, blob, device);
        if (rc != EC_OK) {
            delete m;
            return rc;
        }
        *out = m;
        return EC_OK;
    });
}

/* ============================================== BF16 exponents, rANS top-t codec */
namespace {
/* The exponent table of size up to t from an exponent histogram: exponent 0, then
 * the most frequent other present exponents (ties to the lower one), ascending.
 * rank[e] = index in it, -1 outside. */
int exp_table(const uint64_t hist[256], int t, uint8_t* table, int* rank) {
    bool kept[256] = {};
    kept[0] = true;
    for (int size = 1; size < t; ++size) {
        int best = -1;
        for (int e = 1; e < 256; ++e)
            if (!kept[e] && hist[e] && (best < 0 || hist[e] > hist[best])) best = e;
        if (best < 0) break;
        kept[best] = true;
    }
    int n = 0;
    for (int e = 0; e < 256; ++e) {
        rank[e] = kept[e] ? n : -1;
        if (kept[e]) table[n++] = (uint8_t)e;
    }
    return n;
}

/* Symbol histogram of table size t (symbol = rank, or 16 r0 + r1 for pairs, escapes
 * coded as rank 0) from the exponent histogram (single) or the histogram of the
 * exponent pairs of consecutive lane steps (pairs, 65536 entries); the escape count
 * goes to *esc.  Returns the table size. */
int exp_symbol_hist(bool pair, const uint64_t* hist, const uint64_t* pair_hist, int t, uint8_t* table, int* rank,
                    uint64_t counts[256], uint64_t* esc) {
    const int ts = exp_table(hist, t, table, rank);
    std::fill(counts, counts + 256, uint64_t(0));
    *esc = 0;
    for (int e = 0; e < 256; ++e)
        if (rank[e] < 0) *esc += hist[e];
    if (!pair) {
        for (int e = 0; e < 256; ++e) counts[rank[e] < 0 ? 0 : rank[e]] += hist[e];
    } else {
        for (int e0 = 0; e0 < 256; ++e0)
            for (int e1 = 0; e1 < 256; ++e1) {
                const uint64_t c = pair_hist[e0 * 256 + e1];
                if (c) counts[16 * (rank[e0] < 0 ? 0 : rank[e0]) + (rank[e1] < 0 ? 0 : rank[e1])] += c;
            }
    }
    return ts;
}
}  // namespace

extern "C" int ec_encode_bf16_exp(const uint16_t* w, int64_t n_rows, int64_t k_cols, const ec_exp_params* params,
                                  int device, ec_matrix** out) {
    if (!out) return EC_ERR_INVALID_ARG;
    *out = nullptr;
    if (n_rows < 0 || k_cols < 0) return EC_ERR_SHAPE;
    const int b = params && params->prob_bits ? params->prob_bits : 12;
    const int T = params && params->tile_syms ? params->tile_syms : 4096;
    const bool pair = !params || params->single == 0;
    const int t_req = params ? params->top_t : 0;
    const int t_cap = pair ? 16 : 256;
    if (b < 9 || b > 12 || T < EC_RANS_ROW_ALIGN || T % EC_RANS_ROW_ALIGN || T > 4096 || t_req < 0 || t_req > t_cap ||
        (params && (params->single < 0 || params->single > 1)))
        return EC_ERR_INVALID_ARG;
    if (k_cols > INT64_MAX - EC_RANS_ROW_ALIGN) return EC_ERR_OVERFLOW;
    const int64_t KP = round_up(k_cols, EC_RANS_ROW_ALIGN);
    int64_t nk = 0, n_pad = 0, tmp = 0;
    if (!mul_ok(n_rows, k_cols, &nk) || !mul_ok(n_rows, KP, &n_pad) || !mul_ok(n_pad, 4, &tmp)) return EC_ERR_OVERFLOW;
    if (nk > 0 && !w) return EC_ERR_INVALID_ARG;

    return guarded([&]() -> int {
        const int64_t K = k_cols;
        const int64_t n_tiles = (n_pad + T - 1) / T;
        /* histograms over the padded layout: exponents, and for pairs the exponents of
         * each lane's steps 2m, 2m + 1 (positions 64 m + l and 64 m + 32 + l of a tile) */
        uint64_t hist[256] = {};
        std::vector<uint64_t> pair_hist(pair ? 65536 : 0, 0);
        {
            std::mutex mu;
            parallel_for(n_tiles, [&](int64_t lo, int64_t hi) {
                uint64_t h[256] = {};
                std::vector<uint64_t> ph(pair ? 65536 : 0, 0);
                std::vector<uint16_t> v(T);
                for (int64_t tt = lo; tt < hi; ++tt) {
                    const int64_t base = tt * T, n_t = std::min<int64_t>(T, n_pad - base);
                    gather_padded(w, K, KP, base, n_t, v.data());
                    for (int64_t q = 0; q < n_t; ++q) h[(v[q] >> 7) & 0xFF]++;
                    if (pair)
                        for (int64_t q = 0; q < n_t; q += 64)
                            for (int l = 0; l < 32; ++l) ph[((v[q + l] >> 7) & 0xFF) * 256 + ((v[q + 32 + l] >> 7) & 0xFF)]++;
                }
                std::lock_guard<std::mutex> lk(mu);
                for (int e = 0; e < 256; ++e) hist[e] += h[e];
                for (size_t i = 0; i < ph.size(); ++i) pair_hist[i] += ph[i];
            });
        }
        /* table size: the requested one, or the smallest with the least bound of the
         * coded size (cross-entropy of the stream under the normalised table plus 32
         * bits per escape; MINE section 4.2, "Tuning t") */
        uint8_t table_e[256] = {};
        int rank[256];
        uint64_t counts[256], esc = 0;
        uint32_t freqs[256];
        int t = t_req;
        if (!t) {
            double best = -1.0;
            for (int c = 1; c <= t_cap; ++c) {
                exp_symbol_hist(pair, hist, pair_hist.data(), c, table_e, rank, counts, &esc);
                if (!rans_normalise(counts, 256, b, freqs)) continue;
                double bits = 32.0 * (double)esc;
                for (int s = 0; s < 256; ++s)
                    if (counts[s]) bits += (double)counts[s] * ((double)b - std::log2((double)freqs[s]));
                if (best < 0 || bits < best) {
                    best = bits;
                    t = c;
                }
            }
            if (best < 0) return EC_ERR_INVALID_ARG;
        }
        const int tsize = exp_symbol_hist(pair, hist, pair_hist.data(), t, table_e, rank, counts, &esc);
        ec_matrix* m = new_matrix();
        if (!m) return EC_ERR_OOM;
        std::copy(counts, counts + 256, m->counts);
        if (!rans_normalise(counts, 256, b, m->freqs)) {
            delete m;
            return EC_ERR_INVALID_ARG;
        }
        const uint32_t M = 1u << b;
        uint32_t cum[256];
        for (int s = 0, c = 0; s < 256; ++s) {
            cum[s] = (uint32_t)c;
            c += (int)m->freqs[s];
        }
        /* slot entries: payload (single: the exponent; pair: the symbol) | slot - cum
         * << 8 | freq - 1 << 20; then per pair symbol its two exponent fields */
        std::vector<uint32_t> table(M + 256, 0);
        for (int s = 0; s < 256; ++s)
            for (uint32_t q = 0; q < m->freqs[s]; ++q)
                table[cum[s] + q] = (uint32_t)(pair ? s : table_e[s]) | (q << 8) | ((m->freqs[s] - 1) << 20);
        if (pair)
            for (int r0 = 0; r0 < tsize; ++r0)
                for (int r1 = 0; r1 < tsize; ++r1)
                    table[M + 16 * r0 + r1] = ((uint32_t)table_e[r0] << 7) | ((uint32_t)table_e[r1] << 23);

        const int64_t S_full = T / 32, raw_tile = EC_RAW_BYTES(S_full);
        std::vector<std::vector<uint16_t>> words(n_tiles);
        std::vector<std::vector<uint32_t>> recs(n_tiles);
        std::vector<std::array<uint32_t, 32>> states(n_tiles);
        int64_t raw_total = 0;
        if (!mul_ok(n_tiles, raw_tile, &raw_total)) {
            delete m;
            return EC_ERR_OVERFLOW;
        }
        std::vector<uint8_t> raw((size_t)raw_total, 0);
        const uint64_t unit = uint64_t(1) << (32 - b);
        const int k = pair ? 2 : 1;
        parallel_for(n_tiles, [&](int64_t lo, int64_t hi) {
            std::vector<uint16_t> stack;
            std::vector<uint16_t> v(T);
            for (int64_t tt = lo; tt < hi; ++tt) {
                const int64_t base = tt * T, n_t = std::min<int64_t>(T, n_pad - base), S = n_t / 32;
                gather_padded(w, K, KP, base, n_t, v.data());
                auto rk = [&](int64_t q) {
                    const int r = rank[(v[q] >> 7) & 0xFF];
                    return r < 0 ? 0 : r;
                };
                for (int64_t q = 0; q < n_t; ++q)
                    if (rank[(v[q] >> 7) & 0xFF] < 0) recs[tt].push_back((uint32_t)q | ((uint32_t)v[q] << 16));
                /* sign / mantissa bytes of lane l's symbol i (position 32 i + l) in the
                 * lane-transposed, pair-shuffled layout of the Huffman tiles */
                uint8_t* rt = raw.data() + tt * raw_tile;
                for (int64_t q = 0; q < n_t; ++q) {
                    const int64_t l = q & 31, i = q >> 5;
                    const uint8_t sg = (uint8_t)((v[q] >> 8) & 0x80), mt = (uint8_t)(v[q] & 0x7F);
                    uint8_t* g = rt + ((i >> 4) * 32 + l) * 16 + (i & 12);
                    switch (i & 3) {
                        case 0: g[0] |= mt; g[1] |= sg; break;
                        case 1: g[2] |= mt; g[3] |= sg; break;
                        case 2: g[1] |= mt; g[2] |= sg; break;
                        default: g[3] |= mt; g[0] |= sg; break;
                    }
                }
                uint64_t x[32];
                for (int l = 0; l < 32; ++l) x[l] = 1u << 16;
                stack.clear();
                for (int64_t j = S / k - 1; j >= 0; --j)
                    for (int l = 31; l >= 0; --l) {
                        const int s = pair ? 16 * rk(64 * j + l) + rk(64 * j + 32 + l) : rk(32 * j + l);
                        const uint64_t f = m->freqs[s];
                        if (x[l] >= f * unit) {
                            stack.push_back((uint16_t)x[l]);
                            x[l] >>= 16;
                        }
                        x[l] = ((x[l] / f) << b) + x[l] % f + cum[s];
                    }
                for (int l = 0; l < 32; ++l) states[tt][l] = (uint32_t)x[l];
                words[tt].assign(stack.rbegin(), stack.rend());
            }
        });
        std::vector<uint32_t> tile_off(n_tiles + 1, 0), esc_off(n_tiles + 1, 0);
        int64_t total = 0, max_words = 0, payload = 0, n_esc = 0;
        for (int64_t tt = 0; tt < n_tiles; ++tt) {
            tile_off[tt] = (uint32_t)(total / 16);
            total += 128 + round_up(2 * (int64_t)words[tt].size(), 16);
            max_words = std::max<int64_t>(max_words, (int64_t)words[tt].size());
            payload += 16 * (int64_t)words[tt].size();
            esc_off[tt] = (uint32_t)n_esc;
            n_esc += (int64_t)recs[tt].size();
        }
        if (total / 16 > (int64_t)UINT32_MAX || n_esc > (int64_t)UINT32_MAX) {
            delete m;
            return EC_ERR_OVERFLOW;
        }
        tile_off[n_tiles] = (uint32_t)(total / 16);
        esc_off[n_tiles] = (uint32_t)n_esc;

        ec_blob_header h{};
        h.magic = EC_BLOB_MAGIC;
        h.version = EC_BLOB_VERSION;
        h.kind = EC_KIND_RANS_EXP;
        h.steps = T / 32;
        h.n_rows = n_rows;
        h.k_cols = k_cols;
        h.k_pad = KP;
        h.n_tiles = n_tiles;
        h.table_off = sizeof(ec_blob_header);
        h.table_words = (int64_t)M + 256;
        h.scales_off = round_up(h.table_off + 4 * h.table_words, 16); /* the sign / mantissa section */
        h.tile_off_off = round_up(h.scales_off + raw_total, 16);
        h.esc_off_off = round_up(h.tile_off_off + 4 * (n_tiles + 1), 16);
        h.esc_records_off = round_up(h.esc_off_off + 4 * (n_tiles + 1), 16);
        h.records_off = round_up(h.esc_records_off + 4 * n_esc, 16);
        h.blob_bytes = h.records_off + total;
        h.prob_bits = b;
        h.max_words = (int32_t)max_words;
        h.rans_tuple = k;
        h.fp8_table_size = tsize;
        h.n_escapes = n_esc;

        std::vector<uint8_t> blob((size_t)h.blob_bytes, 0);
        std::memcpy(blob.data(), &h, sizeof h);
        std::memcpy(blob.data() + h.table_off, table.data(), 4 * table.size());
        if (raw_total) std::memcpy(blob.data() + h.scales_off, raw.data(), (size_t)raw_total);
        std::memcpy(blob.data() + h.tile_off_off, tile_off.data(), 4 * tile_off.size());
        std::memcpy(blob.data() + h.esc_off_off, esc_off.data(), 4 * esc_off.size());
        parallel_for(n_tiles, [&](int64_t lo, int64_t hi) {
            for (int64_t tt = lo; tt < hi; ++tt) {
                uint8_t* rec = blob.data() + h.records_off + (int64_t)tile_off[tt] * 16;
                std::memcpy(rec, states[tt].data(), 128);
                if (!words[tt].empty()) std::memcpy(rec + 128, words[tt].data(), 2 * words[tt].size());
                if (!recs[tt].empty())
                    std::memcpy(blob.data() + h.esc_records_off + 4 * (int64_t)esc_off[tt], recs[tt].data(),
                                4 * recs[tt].size());
            }
        });
        m->kind = EC_KIND_RANS_EXP;
        m->device = device;
        m->hdr = h;
        m->payload_bits = payload + 32 * n_esc;
        m->raw_bytes = n_pad;
        m->table_bytes = 4 * h.table_words;
        m->aux_bytes = h.blob_bytes - m->table_bytes - payload / 8 - n_pad;
        m->entropy = entropy_bits(hist, 256); /* bits per exponent */
        int rc = upload(m, blob, device);
        if (rc != EC_OK) {
            delete m;
            return rc;
        }
        *out = m;
        return EC_OK;
    });
}

/* ======================================================= bookkeeping entry points */
extern "C" int ec_stats(const ec_matrix* m, ec_stats_t* s) {
    if (!m || !s) return EC_ERR_INVALID_ARG;
    std::memset(s, 0, sizeof *s);
    s->kind = m->kind;
    s->max_code_len = m->kind == EC_KIND_HUFFMAN_BF16 ? m->hdr.max_len : m->hdr.prob_bits;
    s->n_rows = m->hdr.n_rows;
    s->k_cols = m->hdr.k_cols;
    s->k_pad = m->hdr.k_pad;
    s->n_tiles = m->hdr.n_tiles;
    s->payload_bits = m->payload_bits;
    s->raw_bytes = m->raw_bytes;
    s->aux_bytes = m->aux_bytes;
    s->table_bytes = m->table_bytes;
    s->device_bytes = m->hdr.blob_bytes;
    const double n = (double)m->hdr.n_rows * (double)m->hdr.k_cols;
    s->bits_per_weight = n > 0 ? 8.0 * (double)m->hdr.blob_bytes / n : 0.0;
    s->entropy_bits = m->entropy;
    const double coded = (double)m->hdr.n_rows * (double)m->hdr.k_pad;
    s->coded_bits_per_symbol = coded > 0 ? (double)m->payload_bits / coded : 0.0;
    s->n_records = m->hdr.n_escapes;
    return EC_OK;
}

extern "C" int ec_code_lengths(const ec_matrix* m, uint8_t lengths[256]) {
    if (!m || !lengths) return EC_ERR_INVALID_ARG;
    if (m->kind != EC_KIND_HUFFMAN_BF16) return EC_ERR_UNSUPPORTED;
    std::memcpy(lengths, m->lengths, 256);
    return EC_OK;
}

extern "C" void ec_free(ec_matrix* m) {
    if (!m) return;
    std::free(m->h_blob);
    if (m->d_blob) {
        int prev = 0;
        cudaGetDevice(&prev);
        cudaSetDevice(m->device);
        cudaFree(m->d_blob);
        cudaSetDevice(prev);
    }
    delete m;
}

extern "C" const char* ec_strerror(int code) {
    switch (code) {
        case EC_OK: return "ok";
        case EC_ERR_INVALID_ARG: return "invalid argument";
        case EC_ERR_SHAPE: return "invalid shape";
        case EC_ERR_OVERFLOW: return "size overflow";
        case EC_ERR_UNSUPPORTED: return "unsupported request";
        case EC_ERR_CORRUPT: return "corrupt compressed data";
        case EC_ERR_CUDA: return "CUDA runtime error";
        case EC_ERR_OOM: return "out of memory";
        default: return "unknown error";
    }
}

/* ============================================================ serialisation */
namespace {

struct SerialMeta {
    char magic[8];          /* "ECSER002" */
    int32_t kind, reserved;
    int64_t blob_bytes;
    uint64_t counts[256];
    uint8_t lengths[256];
    uint32_t freqs[256];
    int64_t payload_bits, raw_bytes, aux_bytes, table_bytes;
    double entropy;
};
const char kSerialMagic[8] = {'E', 'C', 'S', 'E', 'R', '0', '0', '2'};

/* Structural validation of a device blob held in host memory: every field and
 * offset is checked with overflow-safe arithmetic before anything trusts it
 * ("M8.9 Quantized Artifacts and Runtime Integration", sections "Parse Before
 * Allocation" and "Container Gates").  Payload bits are not checked here; the
 * kernels bound every read and report EC_ERR_CORRUPT through ec_status. */
int validate_blob(const uint8_t* b, int64_t bytes) {
    if (bytes < (int64_t)sizeof(ec_blob_header)) return EC_ERR_CORRUPT;
    ec_blob_header h;
    std::memcpy(&h, b, sizeof h);
    if (h.magic != EC_BLOB_MAGIC || h.version != EC_BLOB_VERSION) return EC_ERR_CORRUPT;
    if (h.blob_bytes != bytes) return EC_ERR_CORRUPT;
    if (h.kind != EC_KIND_HUFFMAN_BF16 && h.kind != EC_KIND_RANS_INT4 && h.kind != EC_KIND_E8 &&
        h.kind != EC_KIND_RANS_FP8 && h.kind != EC_KIND_RANS_EXP)
        return EC_ERR_CORRUPT;
    if (h.n_rows < 0 || h.k_cols < 0 || h.k_cols > INT64_MAX / 2) return EC_ERR_CORRUPT;
    if (h.kind != EC_KIND_RANS_INT4 && h.rans_values != 0) return EC_ERR_CORRUPT;
    const bool huff = h.kind == EC_KIND_HUFFMAN_BF16, e8 = h.kind == EC_KIND_E8, fp8 = h.kind == EC_KIND_RANS_FP8,
               ex = h.kind == EC_KIND_RANS_EXP;
    const int64_t align = huff ? EC_HUFF_ROW_ALIGN : e8 ? EC_E8_ROW_ALIGN : EC_RANS_ROW_ALIGN;
    if (h.k_pad != round_up(h.k_cols, align)) return EC_ERR_CORRUPT;
    if (e8 ? (h.k_cols % 8 || h.steps < 1 || h.steps > 32)
           : huff ? (h.steps < 16 || h.steps > EC_HUFF_MAX_STEPS || h.steps % 16) : (h.steps < 1 || (32 * h.steps) % align))
        return EC_ERR_CORRUPT;
    int64_t n_pad = 0; /* symbols, or for E8 vectors of 8 weights */
    if (!mul_ok(h.n_rows, e8 ? h.k_pad / 8 : h.k_pad, &n_pad)) return EC_ERR_CORRUPT;
    const int64_t T = 32 * (int64_t)h.steps;
    if (h.n_tiles != (n_pad + T - 1) / T) return EC_ERR_CORRUPT;
    if (h.table_off != (int64_t)sizeof(ec_blob_header)) return EC_ERR_CORRUPT;
    int64_t end = 0, t4 = 0;
    const bool hrec = huff && h.huff_flags == EC_HUFF_WINDOW_REC, recs = fp8 || ex;
    if (huff) {
        if (h.huff_flags != 0 && h.huff_flags != EC_HUFF_WINDOW_REC) return EC_ERR_CORRUPT;
        if (h.huff_sub_tables < 0 || h.huff_sub_tables > 512 || (hrec && h.huff_sub_tables != 0) ||
            h.table_words != EC_PAIR_WORDS + 256 * (int64_t)h.huff_sub_tables)
            return EC_ERR_CORRUPT;
        if (h.max_len < 0 || h.max_len > EC_MAX_CODE_LEN || h.max_code_bytes < 0 || h.max_code_area < 0 ||
            h.max_code_area > h.max_code_bytes)
            return EC_ERR_CORRUPT;
        if (h.window_code_bytes < 0 || h.n_escapes < 0 || (!hrec && h.n_escapes != 0)) return EC_ERR_CORRUPT;
        if (hrec && (32 * (int64_t)h.steps > (int64_t)EC_HREC_POS_MASK + 1 || h.huff_fill < 0 || h.huff_fill > 255))
            return EC_ERR_CORRUPT;
    } else if (e8) {
        if (h.prob_bits < 9 || h.prob_bits > 12 || h.max_words < 0 ||
            h.table_words != (4 * EC_E8_TABLES * EC_E8_ALPHA + ((int64_t)EC_E8_TABLES << h.prob_bits)) / 4)
            return EC_ERR_CORRUPT;
    } else if (fp8) {
        if (h.prob_bits < 9 || h.prob_bits > 12 || h.max_words < 0 || h.rans_tuple != 1 ||
            h.table_words != (int64_t(1) << h.prob_bits) + EC_FP8_VALUE_WORDS || h.fp8_table_size < 1 ||
            h.fp8_table_size > 256 || (32 * (int64_t)h.steps) > 4096 || h.n_escapes < 0)
            return EC_ERR_CORRUPT;
    } else if (ex) {
        if (h.prob_bits < 9 || h.prob_bits > 12 || h.max_words < 0 || (h.rans_tuple != 1 && h.rans_tuple != 2) ||
            h.table_words != (int64_t(1) << h.prob_bits) + 256 || h.fp8_table_size < 1 ||
            h.fp8_table_size > (h.rans_tuple == 2 ? 16 : 256) || (32 * (int64_t)h.steps) > 4096 || h.n_escapes < 0)
            return EC_ERR_CORRUPT;
    } else {
        if (h.prob_bits < 9 || h.prob_bits > 15 || h.table_words != (int64_t(1) << h.prob_bits) || h.max_words < 0)
            return EC_ERR_CORRUPT;
        if (h.rans_tuple != 1 && h.rans_tuple != 2) return EC_ERR_CORRUPT;
        if (h.rans_tuple == 2 && h.prob_bits > 12) return EC_ERR_CORRUPT;
        if (h.rans_values != EC_RANS_VALUES_INT4 && h.rans_values != EC_RANS_VALUES_FP4_E2M1) return EC_ERR_CORRUPT;
    }
    if (!mul_ok(h.table_words, 4, &t4) || !add_ok(h.table_off, t4, &end)) return EC_ERR_CORRUPT;
    if (!huff) { /* rANS: FP16 group scales; E8 and FP8: FP32 row scales; exponents: sign / mantissa bytes */
        int64_t ns = 0, s2 = 0;
        if (ex ? !mul_ok(h.n_tiles, EC_RAW_BYTES(h.steps), &s2)
               : e8 || fp8 ? !mul_ok(h.n_rows, 4, &s2) : (!mul_ok(h.n_rows, h.k_pad / 128, &ns) || !mul_ok(ns, 2, &s2)))
            return EC_ERR_CORRUPT;
        if (h.scales_off < end || h.scales_off % 16 || !add_ok(h.scales_off, s2, &end)) return EC_ERR_CORRUPT;
    }
    int64_t to4 = 0;
    if (h.tile_off_off < end || h.tile_off_off % 16 || !mul_ok(h.n_tiles + 1, 4, &to4) ||
        !add_ok(h.tile_off_off, to4, &end))
        return EC_ERR_CORRUPT;
    if (recs) { /* record offsets, then the records */
        int64_t e4 = 0;
        if (h.esc_off_off < end || h.esc_off_off % 16 || !add_ok(h.esc_off_off, to4, &end)) return EC_ERR_CORRUPT;
        if (h.esc_records_off < end || h.esc_records_off % 16 || !mul_ok(h.n_escapes, 4, &e4) ||
            !add_ok(h.esc_records_off, e4, &end))
            return EC_ERR_CORRUPT;
    }
    if (h.records_off < end || h.records_off % 16 || h.records_off > bytes) return EC_ERR_CORRUPT;
    const uint32_t* off = (const uint32_t*)(b + h.tile_off_off);
    if (off[0] != 0 || (int64_t)off[h.n_tiles] * 16 != bytes - h.records_off) return EC_ERR_CORRUPT;
    int64_t n_hrec = 0; /* Huffman window records seen in the tiles */
    for (int64_t t = 0; t < h.n_tiles; ++t) {
        if (off[t + 1] < off[t]) return EC_ERR_CORRUPT;
        const int64_t rb = ((int64_t)off[t + 1] - off[t]) * 16;
        const int64_t n_t = std::min(T, n_pad - t * T);
        if (huff) {
            /* lane starts (lane 0's slot: the window record count), the code area, the records */
            const int64_t area = rb - 64 - EC_RAW_BYTES(n_t / 32);
            if (area < 16 || area > h.max_code_bytes) return EC_ERR_CORRUPT;
            const uint8_t* tr = b + h.records_off + (int64_t)off[t] * 16;
            const uint16_t* start = (const uint16_t*)tr;
            const int64_t nrec = start[0], code = area - round_up(4 * nrec, 16);
            if ((!hrec && nrec) || code < 16 || code > h.max_code_area) return EC_ERR_CORRUPT;
            for (int l = 1; l < 32; ++l)
                if (start[l] > code || (l > 1 && start[l] < start[l - 1])) return EC_ERR_CORRUPT;
            const uint32_t* rr = (const uint32_t*)(tr + 64 + EC_RAW_BYTES(n_t / 32) + code);
            for (int64_t i = 0; i < nrec; ++i) /* 13-bit positions inside the tile, ascending */
                if ((rr[i] >> (EC_HREC_EXP_SHIFT + 8)) || (int64_t)(rr[i] & EC_HREC_POS_MASK) >= n_t ||
                    (i && (rr[i] & EC_HREC_POS_MASK) <= (rr[i - 1] & EC_HREC_POS_MASK)))
                    return EC_ERR_CORRUPT;
            n_hrec += nrec;
        } else {
            if (rb < 128 || (rb - 128) / 2 > round_up(h.max_words, 8)) return EC_ERR_CORRUPT;
        }
    }
    if (huff && n_hrec != h.n_escapes) return EC_ERR_CORRUPT;
    if (recs) { /* per tile: ascending record offsets, records (position | code << 16) at ascending
                 * positions inside the tile */
        const uint32_t* eo = (const uint32_t*)(b + h.esc_off_off);
        const uint32_t* er = (const uint32_t*)(b + h.esc_records_off);
        if (eo[0] != 0 || (int64_t)eo[h.n_tiles] != h.n_escapes) return EC_ERR_CORRUPT;
        for (int64_t t = 0; t < h.n_tiles; ++t) {
            if (eo[t + 1] < eo[t]) return EC_ERR_CORRUPT;
            const int64_t n_t = std::min(T, n_pad - t * T);
            for (uint32_t e = eo[t]; e < eo[t + 1]; ++e) {
                const uint32_t p = er[e] & 0xFFFFu;
                if ((int64_t)p >= n_t || (fp8 && (er[e] >> 24)) || (e > eo[t] && p <= (er[e - 1] & 0xFFFFu)))
                    return EC_ERR_CORRUPT;
            }
        }
    }
    const uint32_t* tab = (const uint32_t*)(b + h.table_off);
    if (huff) {
        const int64_t n_sub = h.huff_sub_tables;
        for (int64_t i = 0; i < EC_PAIR_WORDS; ++i) { /* pair entries */
            const uint32_t e = tab[i], n = e & EC_PAIR_LEN_MASK, l0 = (e >> EC_PAIR_FIRST_SHIFT) & 15u;
            if ((e & ~EC_PAIR_FIELDS) || l0 > EC_L1_BITS || n > EC_L1_BITS) return EC_ERR_CORRUPT;
            if (!(e & EC_PAIR_OPEN)) { /* complete: two codewords of length >= 1 */
                if (l0 == 0 || n <= l0) return EC_ERR_CORRUPT;
            } else if (l0 > 0) { /* the first codeword only */
                if (n != l0 || ((e >> 23) & 0xFFu) != 0 || (e & 0x8000u)) return EC_ERR_CORRUPT;
            } else { /* a longer first codeword (its sub-table), or no codeword */
                if (n != 0 || ((e >> 23) & 0xFFu) != 0 || (int64_t)((e >> 7) & 0x1FFu) >= std::max<int64_t>(n_sub, 1))
                    return EC_ERR_CORRUPT;
            }
        }
        for (int64_t i = EC_PAIR_WORDS; i < h.table_words; ++i)
            if ((tab[i] & EC_ENT_PTR) && (int64_t)(tab[i] & 0xFFFFu) >= n_sub) return EC_ERR_CORRUPT;
    } else if (e8) { /* per table: frequencies summing to 2^b (or an unused all-zero table), cumulative
                      * starts, and every slot mapped to the symbol whose range holds it */
        const uint32_t M = 1u << h.prob_bits;
        const uint8_t* ss = b + h.table_off + 4 * EC_E8_TABLES * EC_E8_ALPHA;
        for (int t = 0; t < EC_E8_TABLES; ++t) {
            uint32_t c = 0;
            for (int s = 0; s < EC_E8_ALPHA; ++s) {
                const uint32_t e = tab[t * EC_E8_ALPHA + s], f = e & 0xFFFF, cm = e >> 16;
                if (cm != c || f > M) return EC_ERR_CORRUPT;
                for (uint32_t q = 0; q < f; ++q)
                    if (c + q >= M || ss[(size_t)t * M + c + q] != s) return EC_ERR_CORRUPT;
                c += f;
            }
            if (c != M && c != 0) return EC_ERR_CORRUPT;
            if (t == 0 && c != M && n_pad > 0) return EC_ERR_CORRUPT; /* every point has a coset */
            for (int s = 2; t == 0 && s < EC_E8_ALPHA; ++s) /* the coset is 0 or 1 */
                if (tab[s] & 0xFFFFu) return EC_ERR_CORRUPT;
            for (uint32_t q = c; q < M; ++q) /* an unused table maps every slot to symbol 0 */
                if (ss[(size_t)t * M + q] != 0) return EC_ERR_CORRUPT;
        }
    } else if (fp8) { /* pair-layout entries: symbol inside the table, bias below the frequency */
        for (int64_t i = 0; i < (int64_t(1) << h.prob_bits); ++i) {
            const uint32_t f = (tab[i] >> 20) + 1, k = (tab[i] >> 8) & 0xFFF;
            if ((int32_t)(tab[i] & 0xFF) >= h.fp8_table_size || f > (1u << h.prob_bits) || k >= f) return EC_ERR_CORRUPT;
        }
    } else if (ex) { /* pair-layout entries (pair symbols inside the t x t square); the pairs'
                      * exponent fields hold nothing else */
        const uint32_t M = 1u << h.prob_bits, ts = (uint32_t)h.fp8_table_size;
        for (uint32_t i = 0; i < M; ++i) {
            const uint32_t f = (tab[i] >> 20) + 1, k = (tab[i] >> 8) & 0xFFF, s = tab[i] & 0xFF;
            if (f > M || k >= f || (h.rans_tuple == 2 && ((s >> 4) >= ts || (s & 15) >= ts))) return EC_ERR_CORRUPT;
        }
        for (uint32_t i = 0; i < 256; ++i)
            if (tab[M + i] & ~0x7F807F80u) return EC_ERR_CORRUPT;
    } else if (h.rans_tuple == 1) {
        for (int64_t i = 0; i < h.table_words && n_pad > 0; ++i) { /* an empty matrix has an empty table */
            const uint32_t f = tab[i] >> 16, k = (tab[i] >> 4) & 0xFFF;
            if (f == 0 || f > (1u << h.prob_bits) || k >= f) return EC_ERR_CORRUPT;
        }
    } else {
        for (int64_t i = 0; i < h.table_words; ++i) {
            const uint32_t f = (tab[i] >> 20) + 1, k = (tab[i] >> 8) & 0xFFF;
            if (f > (1u << h.prob_bits) || k >= f) return EC_ERR_CORRUPT;
        }
    }
    return EC_OK;
}

}  // namespace

extern "C" int ec_serialize(const ec_matrix* m, void* dst, int64_t capacity, int64_t* size_out) {
    if (!m || !size_out) return EC_ERR_INVALID_ARG;
    const int64_t need = (int64_t)sizeof(SerialMeta) + m->hdr.blob_bytes;
    *size_out = need;
    if (!dst) return EC_OK;
    if (capacity < need) return EC_ERR_INVALID_ARG;
    SerialMeta s{};
    std::memcpy(s.magic, kSerialMagic, 8);
    s.kind = m->kind;
    s.blob_bytes = m->hdr.blob_bytes;
    std::memcpy(s.counts, m->counts, sizeof s.counts);
    std::memcpy(s.lengths, m->lengths, sizeof s.lengths);
    std::memcpy(s.freqs, m->freqs, sizeof s.freqs);
    s.payload_bits = m->payload_bits;
    s.raw_bytes = m->raw_bytes;
    s.aux_bytes = m->aux_bytes;
    s.table_bytes = m->table_bytes;
    s.entropy = m->entropy;
    std::memcpy(dst, &s, sizeof s);
    uint8_t* out = (uint8_t*)dst + sizeof s;
    if (m->h_blob) {
        std::memcpy(out, m->h_blob, (size_t)m->hdr.blob_bytes);
        return EC_OK;
    }
    int prev = 0;
    if (cudaGetDevice(&prev) != cudaSuccess) return EC_ERR_CUDA;
    cudaSetDevice(m->device);
    const cudaError_t e = cudaMemcpy(out, m->d_blob, (size_t)m->hdr.blob_bytes, cudaMemcpyDeviceToHost);
    cudaSetDevice(prev);
    return e == cudaSuccess ? EC_OK : EC_ERR_CUDA;
}

extern "C" int ec_deserialize(const void* src, int64_t size, int device, ec_matrix** out) {
    if (!src || !out) return EC_ERR_INVALID_ARG;
    *out = nullptr;
    if (size < (int64_t)sizeof(SerialMeta)) return EC_ERR_CORRUPT;
    SerialMeta s;
    std::memcpy(&s, src, sizeof s);
    if (std::memcmp(s.magic, kSerialMagic, 8) != 0) return EC_ERR_CORRUPT;
    if (s.blob_bytes < 0 || s.blob_bytes != size - (int64_t)sizeof s) return EC_ERR_CORRUPT;
    const uint8_t* blob = (const uint8_t*)src + sizeof s;
    int rc = validate_blob(blob, s.blob_bytes);
    if (rc != EC_OK) return rc;
    return guarded([&]() -> int {
        ec_matrix* m = new_matrix();
        if (!m) return EC_ERR_OOM;
        std::memcpy(&m->hdr, blob, sizeof m->hdr);
        if (s.kind != m->hdr.kind) {
            delete m;
            return EC_ERR_CORRUPT;
        }
        m->kind = s.kind;
        m->device = device;
        std::memcpy(m->counts, s.counts, sizeof s.counts);
        std::memcpy(m->lengths, s.lengths, sizeof s.lengths);
        std::memcpy(m->freqs, s.freqs, sizeof s.freqs);
        m->payload_bits = s.payload_bits;
        m->raw_bytes = s.raw_bytes;
        m->aux_bytes = s.aux_bytes;
        m->table_bytes = s.table_bytes;
        m->entropy = s.entropy;
        std::vector<uint8_t> copy(blob, blob + s.blob_bytes);
        const int r = upload(m, copy, device);
        if (r != EC_OK) {
            delete m;
            return r;
        }
        *out = m;
        return EC_OK;
    });
}
