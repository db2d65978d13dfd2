// Per-query top-k pool select, expansion to token positions, own tail, -1 pad.
//
// prime-rl PR "GLM-5.3-Flash text model", Summary: a query keeps the top 512
// of the complete pools that end at or before it and also attends to its own
// incomplete pool; index rows are padded to a multiple of 128.  NeMo AutoModel
// PR "add GLM-5.3-Flash training support": 2048 + 3 = 2051 raw slots.
//
// A 256-thread block ranks one query row at a time.  Scores become order-preserving uint32
// keys.  Rows of up to 8192 candidate pools (every row of a document of up to
// 32768 tokens) are ranked from registers on the contiguous path: the row is
// copied into shared memory so that thread t then holds 2-8 consecutive 16-byte
// units (4 pools each, as many as the row length needs) with conflict-free
// loads.  A three-level radix select (bits 31..21, 20..10, 9..0) over the
// registers finds the key K of the topk-th best pool and how many pools equal
// to K still fit; a level whose bin holds exactly the keys still needed is
// kept whole and ends the search.  The kept pools are those with key > K plus
// the first pools with key == K that still fit (lower pool index wins ties).
// One block scan of each thread's count of kept pools gives every thread the
// rank of its first one, and each thread writes its pools' positions in pool
// order, so the row comes out ascending without a sort.  The few rows whose
// copy would not fit the buffer keep the register path (32 keys per thread,
// pools t, t+256, ..., ranked with one ballot per 256-pool column).
//
// Longer rows (documents of more than 32768 tokens) are ranked in chunks of
// 8192 pools: the same levels, and the same compaction chunk by chunk,
// carrying the kept and tied counts from one chunk to the next.  A row of up
// to 16392 pools is first copied whole into shared memory; a longer one is
// read from global memory on every pass, and a pass after level 1 copies the
// keys of the chosen level-1 bin to a shared candidate list that levels 2 and
// 3 then run over.
#include <cstdint>

#include "kpool_common.cuh"
#include "kpool_launch.h"

namespace kpool {

namespace {

constexpr int SEL_THREADS = 256;
constexpr int SEL_WARPS = SEL_THREADS / 32;
constexpr int HIST_BINS = 2048;
constexpr int DECODE_CAND_CAP = 4096;                 // candidate list of the decode select's long rows

// hist also serves as the (column, warp) rank table of the ordered compaction once the radix
// levels are done.
struct SelectSmem {
    uint32_t hist[HIST_BINS];
    int32_t warp_tot[SEL_WARPS];
    uint32_t n_cand;
    uint32_t digit;
    uint32_t remaining;
};

// Exclusive block scan of v (all threads); returns the exclusive prefix and
// writes the block total.
__device__ __forceinline__ int block_excl_scan(int v, int32_t* warp_tot, int& total) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[wid] = x;
    __syncthreads();
    int before = 0;
    total = 0;
#pragma unroll
    for (int w = 0; w < SEL_WARPS; ++w) {
        const int t = warp_tot[w];
        before += (w < wid) ? t : 0;
        total += t;
    }
    __syncthreads();
    return before + x - v;
}

// Finds, in hist[0..nbins), the bin b where the count of keys in bins above b
// is < remaining <= that count + hist[b]; stores b in s.digit and the updated
// remaining (remaining - count above b) in s.remaining.
__device__ void pick_digit(SelectSmem& s, int nbins, uint32_t remaining) {
    const int per = nbins / SEL_THREADS;            // bins per thread (contiguous, descending order)
    const int t = threadIdx.x;
    // thread t owns bins [nbins - (t+1)*per, nbins - t*per), scanned from the top
    int local = 0;
    for (int j = 0; j < per; ++j) local += (int)s.hist[nbins - 1 - (t * per + j)];
    int total;
    const int above = block_excl_scan(local, s.warp_tot, total);
    if ((uint32_t)above < remaining && remaining <= (uint32_t)(above + local)) {
        uint32_t acc = (uint32_t)above;
        for (int j = 0; j < per; ++j) {
            const int b = nbins - 1 - (t * per + j);
            const uint32_t h = s.hist[b];
            if (acc < remaining && remaining <= acc + h) {
                s.digit = (uint32_t)b;
                s.remaining = remaining - acc;
                break;
            }
            acc += h;
        }
    }
    __syncthreads();
}

// Where the positions of a row go: `pool(p)` is the first slot of pool p (the
// pool's 4 positions are consecutive slots), `tok(pos)` the slot of position
// pos of the document or sequence.
// `put(row, rank, p)` writes the 4 slots of pool p as the rank-th kept pool; the checked build
// also verifies that they fall inside the row and the slot range.
struct DocMap {            // packed prefill: slots are global token rows
    int s_d;
    int W, T;
    int32_t* status;
    __device__ __forceinline__ int pool(int p) const { return s_d + KPOOL * p; }
    __device__ __forceinline__ int tok(int pos) const { return s_d + pos; }
    __device__ __forceinline__ void put(int32_t* row, int rank, int p) const {
        const int pos = pool(p);
        if (in_bounds(KPOOL * rank + KPOOL <= W && pos >= 0 && pos + KPOOL <= T, status))
            *reinterpret_cast<int4*>(row + KPOOL * rank) = make_int4(pos, pos + 1, pos + 2, pos + 3);
    }
};
struct PageMap {           // paged decode: 128-token pages listed in the sequence's block table
    const int32_t* bt;
    __device__ __forceinline__ int pool(int p) const { return bt[p >> 5] * 128 + ((KPOOL * p) & 127); }
    __device__ __forceinline__ int tok(int pos) const { return bt[pos >> 7] * 128 + (pos & 127); }
    __device__ __forceinline__ void put(int32_t* row, int rank, int p) const {
        const int pos = pool(p);
        *reinterpret_cast<int4*>(row + KPOOL * rank) = make_int4(pos, pos + 1, pos + 2, pos + 3);
    }
};

constexpr int FAST_KPT = 32;                          // keys per thread on the register path
constexpr int FAST_MAX = SEL_THREADS * FAST_KPT;     // 8192 candidate pools

// One radix level over register-held keys: histogram of bits [shift, shift+log2(nbins)) of the
// keys whose bits above match `prefix` under `hi_mask`, then the digit that holds the
// remaining-th largest key (s.digit, s.remaining).
template <int NC>
__device__ __forceinline__ void fast_level(SelectSmem& s, const uint32_t (&key)[NC], uint32_t hi_mask,
                                           uint32_t prefix, int shift, int nbins, uint32_t remaining) {
    for (int b = threadIdx.x; b < nbins; b += SEL_THREADS) s.hist[b] = 0;
    __syncthreads();
#pragma unroll
    for (int j = 0; j < NC; ++j)
        if ((key[j] & hi_mask) == prefix) atomicAdd(&s.hist[(key[j] >> shift) & (uint32_t)(nbins - 1)], 1u);
    __syncthreads();
    pick_digit(s, nbins, remaining);
}

// Ranks, in pool order, of per-thread flags held as one bit per column: afterwards pool
// 256j + t has rank tab[8j + warp] + popc(ballot of column j & lanes below).  tab (256 entries,
// one per (column, warp) in that order, in s.hist) holds the exclusive scan of the
// per-(column, warp) counts.  The caller reads tab, then synchronises before tab is reused.
// Returns the number of flags set.
template <int NC>
__device__ __forceinline__ int column_scan(SelectSmem& s, uint32_t flags) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    uint32_t* tab = s.hist;                          // the radix levels are done with it
#pragma unroll
    for (int j = 0; j < NC; ++j) {
        const uint32_t b = __ballot_sync(0xffffffffu, (flags >> j) & 1u);
        if (lane == 0) tab[8 * j + wid] = __popc(b);
    }
    __syncthreads();
    int total;
    const int before = block_excl_scan(threadIdx.x < 8 * NC ? (int)tab[threadIdx.x] : 0, s.warp_tot, total);
    tab[threadIdx.x] = (uint32_t)before;
    __syncthreads();
    return total;
}

template <int NC, typename Map>
__device__ void select_registers(SelectSmem& s, const float* __restrict__ sc, int n, int topk, const Map& map,
                                 int32_t* __restrict__ row) {
    const int t = threadIdx.x, wid = t >> 5;
    const uint32_t below = (1u << (t & 31)) - 1u;
    const uint32_t* tab = s.hist;
    uint32_t key[NC];
    // every load first, then the conversions: with sc in global memory (paged decode) the loads
    // are then all in flight together instead of one round trip per key
    float raw[NC];
#pragma unroll
    for (int j = 0; j < NC; ++j) {
        const int p = SEL_THREADS * j + t;
        raw[j] = p < n ? sc[p] : 0.f;
    }
    // Slots past the row (p >= n) get key 0, the key of NaN and the lowest there is, and take part
    // in every count.  They change nothing: with n > topk valid keys the topk-th largest key is
    // that of a valid pool; if it is 0, the slots past the row tie with it at the highest pool
    // indices, so the need_eq lowest-indexed ties are all valid; and the bin of key 0 can never be
    // kept whole (that would need n + the slots past the row <= topk).
#pragma unroll
    for (int j = 0; j < NC; ++j) {
        const int p = SEL_THREADS * j + t;
        key[j] = p < n ? score_key(raw[j]) : 0u;
    }
    // Radix levels over bits 31..21, 20..10, 9..0.  When the bin that holds the
    // topk-th key is kept whole (its count equals the keys still needed), every
    // key from the bin's lowest value up is kept and the later levels are skipped.
    fast_level(s, key, 0u, 0u, 21, 2048, (uint32_t)topk);
    uint32_t prefix = s.digit << 21;
    uint32_t rem = s.remaining, cnt = s.hist[s.digit & 2047u];
    __syncthreads();                                 // every thread has read the bin before it is reused
    bool whole = cnt == rem;
    if (!whole) {
        fast_level(s, key, 0xFFE00000u, prefix, 10, 2048, rem);
        prefix |= s.digit << 10;
        rem = s.remaining;
        cnt = s.hist[s.digit & 2047u];
        __syncthreads();
        whole = cnt == rem;
    }
    uint32_t K = prefix, need_eq = 0, n_eq = 0;      // whole bin: keep every key >= K
    if (!whole) {
        fast_level(s, key, 0xFFFFFC00u, prefix, 0, 1024, rem);
        K = prefix | s.digit;
        need_eq = s.remaining;
        n_eq = s.hist[s.digit & 1023u];              // keys equal to K
        __syncthreads();
    }

    uint32_t gt = 0, eq = 0;
#pragma unroll
    for (int j = 0; j < NC; ++j) {
        gt |= ((whole ? key[j] >= K : key[j] > K) ? 1u : 0u) << j;
        eq |= (!whole && key[j] == K ? 1u : 0u) << j;
    }
    uint32_t take = gt | eq;
    // the column ballots are taken again where the ranks are read: keeping them costs NC registers
    if (n_eq != need_eq) {                           // ties at K: the lowest pool indices among them win
        column_scan<NC>(s, eq);
#pragma unroll
        for (int j = 0; j < NC; ++j) {
            const uint32_t b = __ballot_sync(0xffffffffu, (eq >> j) & 1u);
            if (((eq >> j) & 1u) && tab[8 * j + wid] + __popc(b & below) >= need_eq) take &= ~(1u << j);
        }
        __syncthreads();
    }
    column_scan<NC>(s, take);
#pragma unroll
    for (int j = 0; j < NC; ++j) {
        const uint32_t b = __ballot_sync(0xffffffffu, (take >> j) & 1u);
        const uint32_t rank = tab[8 * j + wid] + __popc(b & below);
        if (((take >> j) & 1u) && rank < (uint32_t)topk) {
            map.put(row, (int)rank, SEL_THREADS * j + t);
        }
    }
}

// Rows of up to 8192 candidates (with the row's offset in its first 16-byte unit) on the
// contiguous path: thread t holds the UPT consecutive 16-byte units t*UPT .. t*UPT+UPT-1 of the
// row, i.e. pools 4*UPT*t - off .. 4*UPT*t - off + 4*UPT - 1 in order (the row was copied into
// shared memory with unit u at position (u % UPT) * 256 + u / UPT, so that these loads are
// conflict-free).  The radix levels are those of the register path; the compaction is one
// block scan of each thread's count of kept pools (and, for ties at K, of its count of ties),
// after which a thread writes its kept pools in order, so the row still comes out ascending.
template <int UPT, typename Map>
__device__ void select_contig(SelectSmem& s, const float* __restrict__ buf, int n, int off, int topk,
                              const Map& map, int32_t* __restrict__ row) {
    constexpr int NC = 4 * UPT;
    const int t = threadIdx.x;
    const int p0 = NC * t - off;                     // pool of this thread's first key
    uint32_t key[NC];
#pragma unroll
    for (int m = 0; m < UPT; ++m) {
        const float4 v = reinterpret_cast<const float4*>(buf)[m * SEL_THREADS + t];
        const float f[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int p = p0 + 4 * m + e;
            // positions outside the row (the first unit's leading floats, the slots past it) get
            // key 0, which changes nothing, as on the register path
            key[4 * m + e] = (p >= 0 && p < n) ? score_key(f[e]) : 0u;
        }
    }
    fast_level(s, key, 0u, 0u, 21, 2048, (uint32_t)topk);
    uint32_t prefix = s.digit << 21;
    uint32_t rem = s.remaining, cnt = s.hist[s.digit & 2047u];
    __syncthreads();
    bool whole = cnt == rem;
    if (!whole) {
        fast_level(s, key, 0xFFE00000u, prefix, 10, 2048, rem);
        prefix |= s.digit << 10;
        rem = s.remaining;
        cnt = s.hist[s.digit & 2047u];
        __syncthreads();
        whole = cnt == rem;
    }
    uint32_t K = prefix, need_eq = 0, n_eq = 0;
    if (!whole) {
        fast_level(s, key, 0xFFFFFC00u, prefix, 0, 1024, rem);
        K = prefix | s.digit;
        need_eq = s.remaining;
        n_eq = s.hist[s.digit & 1023u];
        __syncthreads();
    }
    // Positions outside the row hold key 0: never above K (K > 0 whenever a bin is kept whole), and
    // left out of the ties, which leaves enough valid ties (with n > topk valid pools, fewer than
    // topk keys exceed K = 0) and keeps the leading ones (pool < 0) from being taken first.
    uint32_t gt = 0, eq = 0;
#pragma unroll
    for (int j = 0; j < NC; ++j) {
        gt |= ((whole ? key[j] >= K : key[j] > K) ? 1u : 0u) << j;
        eq |= (!whole && key[j] == K ? 1u : 0u) << j;
    }
    {
        const int lo = p0 < 0 ? -p0 : 0, hi = n - p0 < NC ? n - p0 : NC;   // keys lo .. hi-1 are in the row
        const uint32_t below_hi = hi >= 32 ? 0xFFFFFFFFu : (hi <= 0 ? 0u : (1u << hi) - 1u);
        eq &= below_hi & ~((1u << lo) - 1u);
    }
    uint32_t take = gt;
    if (n_eq != need_eq) {                           // ties at K: the lowest pool indices among them win
        int tot;
        const int before = block_excl_scan(__popc(eq), s.warp_tot, tot);
        uint32_t e = eq;
        for (int k = before; e != 0u && k < (int)need_eq; ++k) {
            take |= e & (0u - e);                    // this thread's next tie, in pool order
            e &= e - 1u;
        }
    } else {
        take |= eq;
    }
    int tot;
    int rank = block_excl_scan(__popc(take), s.warp_tot, tot);
    for (uint32_t b = take; b != 0u && rank < topk; b &= b - 1u, ++rank) {
        map.put(row, rank, p0 + __ffs(b) - 1);
    }
}

}  // namespace

// Keys of chunk c0 (pools c0 + 256j + t in key j) of a row; slots past the row get key 0, as on
// the register path (and for the same reason change nothing).
__device__ __forceinline__ void load_chunk(const float* __restrict__ sc, int n, int c0, uint32_t (&key)[FAST_KPT]) {
    float raw[FAST_KPT];
#pragma unroll
    for (int j = 0; j < FAST_KPT; ++j) {
        const int p = c0 + SEL_THREADS * j + (int)threadIdx.x;
        raw[j] = p < n ? sc[p] : 0.f;
    }
#pragma unroll
    for (int j = 0; j < FAST_KPT; ++j) {
        const int p = c0 + SEL_THREADS * j + (int)threadIdx.x;
        key[j] = p < n ? score_key(raw[j]) : 0u;
    }
}

// One radix level over every chunk of a long row (see fast_level).
__device__ __forceinline__ void chunk_level(SelectSmem& s, const float* __restrict__ sc, int n, uint32_t hi_mask, uint32_t prefix,
                            int shift, int nbins, uint32_t remaining) {
    for (int b = threadIdx.x; b < nbins; b += SEL_THREADS) s.hist[b] = 0;
    __syncthreads();
    for (int c0 = 0; c0 < n; c0 += FAST_MAX) {
        uint32_t key[FAST_KPT];
        load_chunk(sc, n, c0, key);
#pragma unroll
        for (int j = 0; j < FAST_KPT; ++j)
            if ((key[j] & hi_mask) == prefix) atomicAdd(&s.hist[(key[j] >> shift) & (uint32_t)(nbins - 1)], 1u);
    }
    __syncthreads();
    pick_digit(s, nbins, remaining);
}

// One radix level over the candidate list (the keys of the chosen level-1 bin).
__device__ __forceinline__ void list_level(SelectSmem& s, const uint32_t* cand, uint32_t n_list, uint32_t hi_mask,
                                           uint32_t prefix, int shift, int nbins, uint32_t remaining) {
    for (int b = threadIdx.x; b < nbins; b += SEL_THREADS) s.hist[b] = 0;
    __syncthreads();
    for (uint32_t c = threadIdx.x; c < n_list; c += SEL_THREADS) {
        const uint32_t key = cand[c];
        if ((key & hi_mask) == prefix) atomicAdd(&s.hist[(key >> shift) & (uint32_t)(nbins - 1)], 1u);
    }
    __syncthreads();
    pick_digit(s, nbins, remaining);
}

// Rows of more than FAST_MAX candidate pools: the register path's levels and compaction, chunk by
// chunk; sc is in global or shared memory.  After level 1 the keys of the chosen bin are copied to
// `cand` (cand_cap keys; when the bin holds more, or cand is null, levels 2 and 3 re-read the row
// instead).  The compaction walks the chunks in pool order
// with the running count of kept pools (the rank base) and of pools tied at K (which decides the
// ties), and stops once topk pools are kept.
template <typename Map>
__device__ __forceinline__ void select_chunked(SelectSmem& s, uint32_t* cand, int cand_cap,
                                               const float* __restrict__ sc, int n, int topk, const Map& map,
                                               int32_t* __restrict__ row) {
    const int t = threadIdx.x, wid = t >> 5, lane = t & 31;
    const uint32_t below = (1u << lane) - 1u;
    const uint32_t* tab = s.hist;
    chunk_level(s, sc, n, 0u, 0u, 21, 2048, (uint32_t)topk);
    uint32_t prefix = s.digit << 21;
    uint32_t rem = s.remaining, cnt = s.hist[s.digit & 2047u];
    if (t == 0) s.n_cand = 0;
    __syncthreads();
    bool whole = cnt == rem;
    const uint32_t n_list = cnt;                     // keys in the chosen level-1 bin
    const bool listed = cand != nullptr && n_list <= (uint32_t)cand_cap;
    if (!whole && listed) {                          // copy the bin's keys, one atomic per warp and column
        for (int c0 = 0; c0 < n; c0 += FAST_MAX) {
            uint32_t key[FAST_KPT];
            load_chunk(sc, n, c0, key);
#pragma unroll
            for (int j = 0; j < FAST_KPT; ++j) {
                const bool m = (key[j] >> 21) == (prefix >> 21);
                const uint32_t b = __ballot_sync(0xffffffffu, m);
                if (b != 0u) {
                    const int leader = __ffs(b) - 1;
                    uint32_t base = 0;
                    if (lane == leader) base = atomicAdd(&s.n_cand, (uint32_t)__popc(b));
                    base = __shfl_sync(0xffffffffu, base, leader);
                    if (m) cand[base + __popc(b & below)] = key[j];
                }
            }
        }
        __syncthreads();
    }
    if (!whole) {
        if (listed) list_level(s, cand, n_list, 0xFFE00000u, prefix, 10, 2048, rem);
        else chunk_level(s, sc, n, 0xFFE00000u, prefix, 10, 2048, rem);
        prefix |= s.digit << 10;
        rem = s.remaining;
        cnt = s.hist[s.digit & 2047u];
        __syncthreads();
        whole = cnt == rem;
    }
    uint32_t K = prefix, need_eq = 0, n_eq = 0;
    if (!whole) {
        if (listed) list_level(s, cand, n_list, 0xFFFFFC00u, prefix, 0, 1024, rem);
        else chunk_level(s, sc, n, 0xFFFFFC00u, prefix, 0, 1024, rem);
        K = prefix | s.digit;
        need_eq = s.remaining;
        n_eq = s.hist[s.digit & 1023u];
        __syncthreads();
    }
    const bool ties = n_eq != need_eq;
    int sel_base = 0;
    uint32_t eq_base = 0;
    for (int c0 = 0; c0 < n && sel_base < topk; c0 += FAST_MAX) {
        uint32_t key[FAST_KPT];
        load_chunk(sc, n, c0, key);
        uint32_t gt = 0, eq = 0;
#pragma unroll
        for (int j = 0; j < FAST_KPT; ++j) {
            gt |= ((whole ? key[j] >= K : key[j] > K) ? 1u : 0u) << j;
            eq |= (!whole && key[j] == K ? 1u : 0u) << j;
        }
        uint32_t take = gt | eq;
        if (ties) {                                  // the lowest pool indices among the ties win
            const int eq_tot = column_scan<FAST_KPT>(s, eq);
#pragma unroll
            for (int j = 0; j < FAST_KPT; ++j) {
                const uint32_t b = __ballot_sync(0xffffffffu, (eq >> j) & 1u);
                if (((eq >> j) & 1u) && eq_base + tab[8 * j + wid] + __popc(b & below) >= need_eq)
                    take &= ~(1u << j);
            }
            __syncthreads();
            eq_base += (uint32_t)eq_tot;
        }
        const int take_tot = column_scan<FAST_KPT>(s, take);
#pragma unroll
        for (int j = 0; j < FAST_KPT; ++j) {
            const uint32_t b = __ballot_sync(0xffffffffu, (take >> j) & 1u);
            const int rank = sel_base + (int)(tab[8 * j + wid] + __popc(b & below));
            if (((take >> j) & 1u) && rank < topk) {
                map.put(row, rank, c0 + SEL_THREADS * j + t);
            }
        }
        __syncthreads();                             // tab is reused by the next chunk
        sel_base += take_tot;
    }
}


// Row metadata: document, in-document position, candidate count and the
// element offset of the row's scores in the compact triangle.
struct RowInfo {
    int d, s_d, r, n, tail;
    int64_t start;
};

__device__ __forceinline__ RowInfo row_info(int i, const int64_t* __restrict__ pair_base,
                                            const int32_t* __restrict__ cu_seqlens,
                                            const int32_t* __restrict__ cu_pools, const int32_t* __restrict__ tok_doc,
                                            int n_docs) {
    RowInfo ri;
    ri.d = (cu_pools[n_docs] < 0) ? -1 : tok_doc[i];
    ri.s_d = ri.r = ri.n = ri.tail = 0;
    ri.start = 0;
    if (ri.d >= 0) {
        ri.s_d = cu_seqlens[ri.d];
        ri.r = i - ri.s_d;
        ri.n = (ri.r + 1) / KPOOL;
        ri.tail = (ri.r + 1) % KPOOL;
        ri.start = pair_base[ri.d] + pairs_before(ri.r);
    }
    return ri;
}

constexpr int ROWBUF = FAST_MAX + 8;                  // floats per row buffer (+ alignment slack)

// Asynchronous copy of a row's n scores into `buf` (16-byte units from the unit
// holding the first score; the last unit copies only the bytes of the row).
// The first score is buf[start % 4].
__device__ __forceinline__ void prefetch_row(float* buf, const float* __restrict__ scores, int64_t start, int n) {
    const int64_t b0 = start * 4, b1 = (start + n) * 4;
    const int64_t u0 = b0 >> 4, u1 = (b1 + 15) >> 4;
    const char* base = reinterpret_cast<const char*>(scores);
    const uint32_t dst0 = static_cast<uint32_t>(__cvta_generic_to_shared(buf));
    for (int64_t u = u0 + threadIdx.x; u < u1; u += SEL_THREADS) {
        const int64_t off = u * 16;
        const int64_t rem = b1 - off;
        const uint32_t bytes = rem < 16 ? (uint32_t)rem : 16u;
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst0 + (uint32_t)(u - u0) * 16u),
                     "l"(base + off), "r"(bytes)
                     : "memory");
    }
}

// Units per thread of the contiguous path for a row of n scores starting at float offset
// start % 4 of its first unit (2, 3, 4, 6 or 8), or 0 when the row takes the register path.
__device__ __forceinline__ int contig_upt(int64_t start, int n) {
    const int f = n + (int)(start & 3);              // floats copied
    if (f <= 2048) return 2;
    if (f <= 3072) return 3;
    if (f <= 4096) return 4;
    if (f <= 6144) return 6;
    if (f <= 8192) return 8;
    return 0;
}

// As prefetch_row, with unit u of the row at position (u % upt) * 256 + u / upt of the buffer.
__device__ __forceinline__ void prefetch_row_contig(float* buf, const float* __restrict__ scores, int64_t start,
                                                    int n, int upt) {
    const int64_t b0 = start * 4, b1 = (start + n) * 4;
    const int64_t u0 = b0 >> 4, u1 = (b1 + 15) >> 4;
    const char* base = reinterpret_cast<const char*>(scores);
    const uint32_t dst0 = static_cast<uint32_t>(__cvta_generic_to_shared(buf));
    for (int64_t u = u0 + threadIdx.x; u < u1; u += SEL_THREADS) {
        const int64_t off = u * 16;
        const int64_t rem = b1 - off;
        const uint32_t bytes = rem < 16 ? (uint32_t)rem : 16u;
        const int ur = (int)(u - u0);
        const uint32_t posn = (uint32_t)((ur % upt) * SEL_THREADS + ur / upt);
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst0 + posn * 16u), "l"(base + off),
                     "r"(bytes)
                     : "memory");
    }
}

__device__ __forceinline__ bool fast_row(const RowInfo& ri, int topk) {
    return ri.d >= 0 && ri.n > topk && ri.n <= FAST_MAX;
}

constexpr int MID_MAX = 2 * ROWBUF - 8;               // pools of a row that fits both row buffers

__device__ __forceinline__ bool mid_row(const RowInfo& ri, int topk) {
    return ri.d >= 0 && ri.n > topk && ri.n > FAST_MAX && ri.n <= MID_MAX;
}

constexpr int SEL_CTAS_PER_SM = 3;                   // 3 x (65.6 KB row buffers + 8.2 KB) of shared memory

// Persistent: block b walks rows row0 + b, row0 + b + gridDim.x, ... below row1; the scores of the
// next row are copied into shared memory (cp.async) while the current row is
// ranked, so the load latency of a row is hidden behind the previous one.
// A row longer than one row buffer but not two is copied into both when its
// turn comes (the next row's copy then starts after it); longer rows are read
// from global memory.
__global__ void __launch_bounds__(SEL_THREADS, SEL_CTAS_PER_SM) select_kernel(const float* __restrict__ scores,
                                                             const int64_t* __restrict__ pair_base,
                                                             const int32_t* __restrict__ cu_seqlens,
                                                             const int32_t* __restrict__ cu_pools,
                                                             const int32_t* __restrict__ tok_doc, int n_docs, int T,
                                                             int topk, int32_t* __restrict__ indices, int W,
                                                             int64_t n_scores, int32_t* status, int row0,
                                                             int row1) {
    __shared__ SelectSmem s;
    extern __shared__ __align__(16) float rowbuf[];   // 2 x ROWBUF
    const int t = threadIdx.x;
    int i = row0 + (int)blockIdx.x;                   // rows row0 .. row1-1 (row1 <= T)
    if (i >= row1) return;
    // checked build: a row whose scores would fall outside the score triangle is left empty
    auto scores_ok = [&](RowInfo& ri) {
        if (ri.d >= 0 && ri.n > topk && !in_bounds(ri.start >= 0 && ri.start + ri.n <= n_scores, status)) ri.d = -1;
    };
    RowInfo cur = row_info(i, pair_base, cu_seqlens, cu_pools, tok_doc, n_docs);
    scores_ok(cur);
    if (fast_row(cur, topk)) {
        const int upt = contig_upt(cur.start, cur.n);
        if (upt) prefetch_row_contig(rowbuf, scores, cur.start, cur.n, upt);
        else prefetch_row(rowbuf, scores, cur.start, cur.n);
    }
    asm volatile("cp.async.commit_group;\n" ::: "memory");
    for (int k = 0; i < row1; ++k, i += gridDim.x) {
        const int i2 = i + (int)gridDim.x;
        RowInfo nxt;
        nxt.d = -1;
        if (i2 < row1) {
            nxt = row_info(i2, pair_base, cu_seqlens, cu_pools, tok_doc, n_docs);
            scores_ok(nxt);
        }
        const bool cur_mid = mid_row(cur, topk);
        const bool pf_nxt = fast_row(nxt, topk);
        if (pf_nxt && !cur_mid) {
            const int upt = contig_upt(nxt.start, nxt.n);
            if (upt) prefetch_row_contig(rowbuf + ((k + 1) & 1) * ROWBUF, scores, nxt.start, nxt.n, upt);
            else prefetch_row(rowbuf + ((k + 1) & 1) * ROWBUF, scores, nxt.start, nxt.n);
        }
        asm volatile("cp.async.commit_group;\n" ::: "memory");

        int32_t* row = indices + (int64_t)i * W;
        const DocMap map{cur.s_d, W, T, status};
        if (cur.d < 0) {
            for (int j = t; j < W; j += SEL_THREADS) row[j] = -1;
        } else if (cur.n <= topk) {                   // every candidate is kept: the causal prefix
            for (int j = t; j < W; j += SEL_THREADS) row[j] = (j <= cur.r) ? map.tok(j) : -1;
        } else {
            if (cur.n <= FAST_MAX) {
                asm volatile("cp.async.wait_group 1;\n" ::: "memory");
                __syncthreads();
                const float* bufk = rowbuf + (k & 1) * ROWBUF;
                const int off = (int)(cur.start & 3);
                switch (contig_upt(cur.start, cur.n)) {
                    case 2: select_contig<2>(s, bufk, cur.n, off, topk, map, row); break;
                    case 3: select_contig<3>(s, bufk, cur.n, off, topk, map, row); break;
                    case 4: select_contig<4>(s, bufk, cur.n, off, topk, map, row); break;
                    case 6: select_contig<6>(s, bufk, cur.n, off, topk, map, row); break;
                    case 8: select_contig<8>(s, bufk, cur.n, off, topk, map, row); break;
                    default: select_registers<32>(s, bufk + off, cur.n, topk, map, row); break;
                }
            } else if (cur_mid) {                     // no copy is in flight: this row was not prefetched
                prefetch_row(rowbuf, scores, cur.start, cur.n);
                asm volatile("cp.async.commit_group;\n" ::: "memory");
                asm volatile("cp.async.wait_group 0;\n" ::: "memory");
                __syncthreads();
                select_chunked(s, nullptr, 0, rowbuf + (int)(cur.start & 3), cur.n, topk, map, row);
            } else {
                // a row too long for the row buffers leaves its own buffer free for the candidate list
                uint32_t* cand = reinterpret_cast<uint32_t*>(rowbuf + (k & 1) * ROWBUF);
                select_chunked(s, cand, FAST_MAX, scores + cur.start, cur.n, topk, map, row);
            }
            for (int j = KPOOL * topk + t; j < W; j += SEL_THREADS) {
                const int q = j - KPOOL * topk;
                row[j] = q < cur.tail ? map.tok(cur.r - cur.tail + 1 + q) : -1;
            }
        }
        __syncthreads();                              // the row buffer and s are reused
        if (pf_nxt && cur_mid) prefetch_row(rowbuf + ((k + 1) & 1) * ROWBUF, scores, nxt.start, nxt.n);
        asm volatile("cp.async.commit_group;\n" ::: "memory");
        cur = nxt;
    }
    asm volatile("cp.async.wait_group 0;\n" ::: "memory");
}

// Paged decode: one block per sequence b, whose query is its last token
// (position r = seq_lens[b] - 1).  Its n = seq_lens[b] / 4 complete pools have
// scores at scores[b * stride + p]; positions map to latent-cache slots through
// the sequence's row of the block table.
__global__ void __launch_bounds__(SEL_THREADS, 2) decode_select_kernel(const float* __restrict__ scores, int64_t stride,
                                                                    const int32_t* __restrict__ seq_lens,
                                                                    const int32_t* __restrict__ block_table,
                                                                    int max_pages, int topk,
                                                                    int32_t* __restrict__ indices, int W) {
    __shared__ SelectSmem s;
    __shared__ uint32_t cand[DECODE_CAND_CAP];
    const int t = threadIdx.x, b = blockIdx.x;
    const int L = seq_lens[b];
    int32_t* row = indices + (int64_t)b * W;
    const PageMap map{block_table + (int64_t)b * max_pages};
    const int r = L - 1, n = L / KPOOL, tail = L % KPOOL;
    const float* sc = scores + (int64_t)b * stride;
    if (L <= 0 || L > max_pages * 128) {              // empty, or more than the block table holds
        for (int j = t; j < W; j += SEL_THREADS) row[j] = -1;
    } else if (n <= topk) {
        for (int j = t; j < W; j += SEL_THREADS) row[j] = (j <= r) ? map.tok(j) : -1;
    } else {
        if (n <= 8 * SEL_THREADS) select_registers<8>(s, sc, n, topk, map, row);
        else if (n <= 16 * SEL_THREADS) select_registers<16>(s, sc, n, topk, map, row);
        else if (n <= FAST_MAX) select_registers<32>(s, sc, n, topk, map, row);
        else select_chunked(s, cand, DECODE_CAND_CAP, sc, n, topk, map, row);
        for (int j = KPOOL * topk + t; j < W; j += SEL_THREADS) {
            const int q = j - KPOOL * topk;
            row[j] = q < tail ? map.tok(r - tail + 1 + q) : -1;
        }
    }
}

int launch_decode_select(const float* scores, int64_t stride, const int32_t* seq_lens, const int32_t* block_table,
                         int max_pages, int B, int topk, int32_t* indices, int W, cudaStream_t stream) {
    if (B <= 0) return KPOOL_OK;
    decode_select_kernel<<<B, SEL_THREADS, 0, stream>>>(scores, stride, seq_lens, block_table, max_pages, topk,
                                                        indices, W);
    return cudaGetLastError() == cudaSuccess ? KPOOL_OK : KPOOL_ERR_CUDA;
}

int launch_select(const float* scores, const int64_t* pair_base, const kpool_layout& L, int topk, int32_t* indices,
                  int W, cudaStream_t stream, int row0, int row1) {
    if (row1 < 0 || row1 > L.T) row1 = L.T;
    if (row0 < 0) return KPOOL_ERR_INVALID_ARG;
    if (row0 >= row1) return KPOOL_OK;
    constexpr int kDyn = 2 * ROWBUF * (int)sizeof(float);
    static int n_sm[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return KPOOL_ERR_CUDA;
    if (n_sm[dev] == 0) {
        if (cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDyn) != cudaSuccess)
            return KPOOL_ERR_CUDA;
        // the whole carveout as shared memory, so SEL_CTAS_PER_SM blocks fit on an SM
        if (cudaFuncSetAttribute(select_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100) != cudaSuccess)
            return KPOOL_ERR_CUDA;
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return KPOOL_ERR_CUDA;
        n_sm[dev] = sms;
    }
    const int n = row1 - row0;
    const int grid = n < SEL_CTAS_PER_SM * n_sm[dev] ? n : SEL_CTAS_PER_SM * n_sm[dev];
    select_kernel<<<grid, SEL_THREADS, kDyn, stream>>>(scores, pair_base, L.cu_seqlens, L.cu_pools, L.tok_doc,
                                                      L.n_docs, L.T, topk, indices, W, pairs_before(L.T), L.status,
                                                      row0, row1);
    return cudaGetLastError() == cudaSuccess ? KPOOL_OK : KPOOL_ERR_CUDA;
}

}  // namespace kpool
