/*
 * Body of the CPU oracle, written once and included twice by det_oracle.c
 * with T = float / SFX = f32 and T = double / SFX = f64, SCAN_E = elements
 * per virtual lane of a scan chunk.
 *
 * TEST INFRASTRUCTURE ONLY.  Every loop here is the plain, sequential
 * statement of the association order the library promises; nothing is
 * blocked, fused or reordered.  IEEE arithmetic in the input's own precision
 * (the pages fix Float32/Float64), round to nearest, no contraction (there
 * are no multiplies), no flush-to-zero.
 */

#define CAT_(a, b) a##_##b
#define CAT(a, b) CAT_(a, b)
#define FN(name) CAT(name, SFX)

/* "absent" term: x + (-0.0) == x bit-exactly for every x under round to
 * nearest, so an absent operand is the same as passing the other one through. */
#define ABSENT ((T)-0.0)

/* ---------------------------------------------------------------------- */
/* PT: the canonical pairwise tree over v[0..m), m >= 1.
 *
 * Definition: pad v with absent terms to the next power of two P and add the
 * perfect binary tree level by level, pairing (2j, 2j+1).  The root splits the
 * padded range at P/2, which is the largest power of two below m, so the
 * recursion below is that definition read top-down.  The bracket depends on
 * element index only, never on how many threads or blocks compute it.
 * (Day 68 "Floating point and reproducibility", section "Contracts from
 *  tolerance to fixed bits", item 1 and the ten-round tree figure: a fixed
 *  pairing of partials; here the pairing is frozen by index instead of by
 *  the grid, see item 2 of the same section.) */
static T FN(pt)(const T* v, int64_t m)
{
    if (m == 1) return v[0];
    int64_t h = 1;
    while (h * 2 < m) h *= 2;
    T left = FN(pt)(v, h);
    T right = FN(pt)(v + h, m - h);
    return left + right;
}

/* ---------------------------------------------------------------------- */
/* det_sum: PT(x[0..n)); the empty sum is +0.0. */
int FN(oracle_sum)(const T* x, int64_t n, T* out)
{
    if (n < 0 || !out || (n > 0 && !x)) return 1;
    *out = (n == 0) ? (T)0.0 : FN(pt)(x, n);
    return 0;
}

/* ---------------------------------------------------------------------- */
/* det_scatter_add: out[bins[i]] += values[i] for every valid i, as
 *   1. records (bins[i], values[i], i) for valid i (0 <= bins[i] < m; other
 *      indices are skipped, as tile_atomic_add_indexed skips negative and
 *      past-the-end destinations);
 *   2. a stable sort by destination, so each group keeps ascending i
 *      (Warp "Deterministic Execution", "Pattern 1: Accumulation" and
 *      "Picking the Right Mode": sort by destination and linear thread index);
 *   3. each non-empty group reduced by PT over its values in that order, and
 *      the old value added once, last: out[b] = out[b] + PT(group).
 * Groups with no element leave out[b] untouched.
 * perm_out (n entries, may be NULL) receives the sorted record indices;
 * seg_offsets_out (m+1 entries, may be NULL) the group starts. */
int FN(oracle_scatter_add)(T* out, int64_t m, const int32_t* bins, const T* values,
                           int64_t n, int32_t* perm_out, int32_t* seg_offsets_out)
{
    if (m < 0 || n < 0 || (m > 0 && !out) || (n > 0 && (!bins || !values))) return 1;
    if (n > 2147483647LL || m > 2147483647LL) return 2;
    int64_t* count = (int64_t*)calloc((size_t)m + 1, sizeof(int64_t));
    if (!count) return 3;
    for (int64_t i = 0; i < n; ++i) {
        int64_t b = bins[i];
        if (b >= 0 && b < m) count[b] += 1;
    }
    /* group starts: exclusive prefix of the counts */
    int64_t* start = (int64_t*)malloc(((size_t)m + 1) * sizeof(int64_t));
    int64_t* cursor = (int64_t*)malloc(((size_t)m + 1) * sizeof(int64_t));
    int64_t total = 0;
    for (int64_t b = 0; b < m; ++b) { start[b] = total; total += count[b]; }
    start[m] = total;
    int32_t* perm = (int32_t*)malloc(((size_t)total + 1) * sizeof(int32_t));
    for (int64_t b = 0; b <= m; ++b) cursor[b] = start[b];
    /* stable placement: ascending i within each destination */
    for (int64_t i = 0; i < n; ++i) {
        int64_t b = bins[i];
        if (b >= 0 && b < m) perm[cursor[b]++] = (int32_t)i;
    }
    T* tmp = (T*)malloc(((size_t)total + 1) * sizeof(T));
    for (int64_t b = 0; b < m; ++b) {
        int64_t len = count[b];
        if (len == 0) continue;
        for (int64_t r = 0; r < len; ++r) tmp[r] = values[perm[start[b] + r]];
        T group = FN(pt)(tmp, len);
        out[b] = out[b] + group;
    }
    if (perm_out) for (int64_t k = 0; k < total; ++k) perm_out[k] = perm[k];
    if (seg_offsets_out) for (int64_t b = 0; b <= m; ++b) seg_offsets_out[b] = (int32_t)start[b];
    free(tmp); free(perm); free(cursor); free(start); free(count);
    return 0;
}

/* ---------------------------------------------------------------------- */
/* det_scatter_sub: the deterministic form of wp.atomic_sub(out, bins[i],
 * values[i]).  The values are negated and then added in det_scatter_add's
 * fixed order: out[b] = out[b] + PT(-values of group b), groups as above
 * (Warp "Deterministic Execution", "Pattern 1: Accumulation", table row
 * atomic_sub: values are negated and added in a fixed order). */
int FN(oracle_scatter_sub)(T* out, int64_t m, const int32_t* bins, const T* values, int64_t n)
{
    if (n < 0 || (n > 0 && !values)) return 1;
    T* neg = (T*)malloc(((size_t)n + 1) * sizeof(T));
    if (!neg) return 3;
    for (int64_t i = 0; i < n; ++i) neg[i] = -values[i];
    int rc = FN(oracle_scatter_add)(out, m, bins, neg, n, NULL, NULL);
    free(neg);
    return rc;
}

/* IEEE 754-2019 minimum / maximum: a NaN operand gives NaN (returned as the
 * canonical quiet NaN: payloads are not promised), -0 orders below +0, else
 * the smaller / larger operand.  Both are associative and commutative, so a
 * group's result does not depend on the order it is combined in. */
static T FN(ieee_minimum)(T a, T b)
{
    if (a != a || b != b) return (T)NAN;
    if (a == b) return signbit(a) ? a : b;
    return a < b ? a : b;
}
static T FN(ieee_maximum)(T a, T b)
{
    if (a != a || b != b) return (T)NAN;
    if (a == b) return signbit(a) ? b : a;
    return a > b ? a : b;
}

/* det_scatter_min / det_scatter_max: the deterministic form of
 * wp.atomic_min / wp.atomic_max(out, bins[i], values[i]): values are grouped
 * by destination and minimized (maximized), and the old value takes part:
 * out[b] = op(out[b], op over group b) for non-empty groups; other entries
 * are untouched (Warp "Deterministic Execution", "Pattern 1: Accumulation",
 * table rows atomic_min and atomic_max).  Invalid bins are skipped as in
 * det_scatter_add.  is_max selects the maximum. */
int FN(oracle_scatter_minmax)(T* out, int64_t m, const int32_t* bins, const T* values, int64_t n, int is_max)
{
    if (m < 0 || n < 0 || (m > 0 && !out) || (n > 0 && (!bins || !values))) return 1;
    if (n > 2147483647LL || m > 2147483647LL) return 2;
    T* acc = (T*)malloc(((size_t)m + 1) * sizeof(T));
    unsigned char* seen = (unsigned char*)calloc((size_t)m + 1, 1);
    if (!acc || !seen) { free(acc); free(seen); return 3; }
    for (int64_t i = 0; i < n; ++i) {   /* index order; any order gives the same result */
        int64_t b = bins[i];
        if (b < 0 || b >= m) continue;
        if (!seen[b]) { acc[b] = values[i]; seen[b] = 1; continue; }
        acc[b] = is_max ? FN(ieee_maximum)(acc[b], values[i]) : FN(ieee_minimum)(acc[b], values[i]);
    }
    for (int64_t b = 0; b < m; ++b)
        if (seen[b]) out[b] = is_max ? FN(ieee_maximum)(out[b], acc[b]) : FN(ieee_minimum)(out[b], acc[b]);
    free(acc); free(seen);
    return 0;
}

/* ---------------------------------------------------------------------- */
/* det_scatter_add_rows: the tile row scatter of warp.tile_atomic_add_indexed
 * (axis 0): source row s is added to destination row idx[s] + row_offset;
 * destinations outside [0, dst_rows) are skipped; repeated rows accumulate.
 * Column by column this is exactly det_scatter_add: the rows aimed at one
 * destination are taken in ascending s and reduced by PT, then added once to
 * the old row.  prev_out[s] (may be NULL) receives the destination row as it
 * was before this call for every valid s, and +0.0 for skipped rows. */
int FN(oracle_scatter_add_rows)(T* dst, int64_t dst_rows, int64_t row_len,
                                const int32_t* idx, int64_t row_offset,
                                const T* src, int64_t src_rows, T* prev_out)
{
    if (dst_rows < 0 || row_len < 0 || src_rows < 0) return 1;
    if (src_rows > 0 && (!idx || (row_len > 0 && !src))) return 1;
    if (dst_rows > 0 && row_len > 0 && !dst) return 1;
    if (src_rows > 2147483647LL || dst_rows > 2147483647LL) return 2;
    int64_t R = dst_rows, W = row_len, M = src_rows;
    T* old = (T*)malloc(((size_t)(R * W) + 1) * sizeof(T));
    for (int64_t k = 0; k < R * W; ++k) old[k] = dst[k];
    int64_t* count = (int64_t*)calloc((size_t)R + 1, sizeof(int64_t));
    for (int64_t s = 0; s < M; ++s) {
        int64_t r = (int64_t)idx[s] + row_offset;
        if (r >= 0 && r < R) count[r] += 1;
    }
    int64_t* start = (int64_t*)malloc(((size_t)R + 1) * sizeof(int64_t));
    int64_t* cursor = (int64_t*)malloc(((size_t)R + 1) * sizeof(int64_t));
    int64_t total = 0;
    for (int64_t r = 0; r < R; ++r) { start[r] = total; total += count[r]; }
    start[R] = total;
    int32_t* perm = (int32_t*)malloc(((size_t)total + 1) * sizeof(int32_t));
    for (int64_t r = 0; r <= R; ++r) cursor[r] = start[r];
    for (int64_t s = 0; s < M; ++s) {
        int64_t r = (int64_t)idx[s] + row_offset;
        if (r >= 0 && r < R) perm[cursor[r]++] = (int32_t)s;
    }
    T* tmp = (T*)malloc(((size_t)total + 1) * sizeof(T));
    for (int64_t r = 0; r < R; ++r) {
        int64_t len = count[r];
        if (len == 0) continue;
        for (int64_t j = 0; j < W; ++j) {
            for (int64_t k = 0; k < len; ++k) tmp[k] = src[(int64_t)perm[start[r] + k] * W + j];
            T group = FN(pt)(tmp, len);
            dst[r * W + j] = old[r * W + j] + group;
        }
    }
    if (prev_out) {
        for (int64_t s = 0; s < M; ++s) {
            int64_t r = (int64_t)idx[s] + row_offset;
            for (int64_t j = 0; j < W; ++j)
                prev_out[s * W + j] = (r >= 0 && r < R) ? old[r * W + j] : (T)0.0;
        }
    }
    free(tmp); free(perm); free(cursor); free(start); free(count); free(old);
    return 0;
}

/* det_scatter_add_rows_ordered: the same row scatter with the tile page's
 * "returns the previous value" read as atomics applied one source row at a
 * time in ascending s: per destination row and column the contributions are
 * added sequentially to the old value, prev_out[s] receives the running value
 * just before row s is added, and the destination ends at the full
 * sequential sum (Warp language reference "warp.tile_atomic_add_indexed",
 * returns; the index-order running prefix per destination).  Skipped rows get
 * prev +0.0 as in det_scatter_add_rows. */
int FN(oracle_scatter_add_rows_ordered)(T* dst, int64_t dst_rows, int64_t row_len,
                                        const int32_t* idx, int64_t row_offset,
                                        const T* src, int64_t src_rows, T* prev_out)
{
    if (dst_rows < 0 || row_len < 0 || src_rows < 0) return 1;
    if (src_rows > 0 && (!idx || (row_len > 0 && !src))) return 1;
    if (dst_rows > 0 && row_len > 0 && !dst) return 1;
    if (src_rows > 2147483647LL || dst_rows > 2147483647LL) return 2;
    const int64_t R = dst_rows, W = row_len, M = src_rows;
    for (int64_t s = 0; s < M; ++s) {          /* ascending source row: thread order */
        const int64_t r = (int64_t)idx[s] + row_offset;
        for (int64_t j = 0; j < W; ++j) {
            if (r < 0 || r >= R) {
                if (prev_out) prev_out[s * W + j] = (T)0.0;
                continue;
            }
            if (prev_out) prev_out[s * W + j] = dst[r * W + j];
            dst[r * W + j] = dst[r * W + j] + src[s * W + j];
        }
    }
    return 0;
}

/* det_gather_rows: out[i] = src[idx[i] + row_offset] row by row, +0.0 for
 * indices outside [0, src_rows) -- the forward gather of Warp "Deterministic
 * Execution", "Tape and Backward Passes" (out[tid] = values[indices[tid]]),
 * whose adjoint is det_scatter_add_rows of the output gradient. */
int FN(oracle_gather_rows)(T* out, const T* src, int64_t src_rows, int64_t row_len, const int32_t* idx,
                           int64_t row_offset, int64_t n)
{
    if (src_rows < 0 || row_len < 0 || n < 0) return 1;
    if (n > 0 && row_len > 0 && (!out || !idx || (src_rows > 0 && !src))) return 1;
    for (int64_t i = 0; i < n; ++i) {
        const int64_t r = (int64_t)idx[i] + row_offset;
        for (int64_t j = 0; j < row_len; ++j)
            out[i * row_len + j] = (r >= 0 && r < src_rows) ? src[r * row_len + j] : (T)0.0;
    }
    return 0;
}

/* ---------------------------------------------------------------------- */
/* Anchored decoupled look-back scan (drjit-core pull request "Make CUDA
 * floating-point prefix sums deterministic", sections "Implementation" and
 * the reworked description in the follow-up comment).
 *
 * The input is cut into chunks of C = NWARP * NLANE * SCAN_E elements.  Inside
 * chunk c element t = w*NLANE*E + l*E + e belongs to virtual lane l of virtual
 * warp w.  Elements past n are absent.
 *
 *   lane total   LT[w][l] = ((x0 + x1) + x2) + ... + x(E-1)     (in-lane fold)
 *   lane prefix  Kogge-Stone over l: K[l] = K[l-2^r] + K[l] for l >= 2^r,
 *                r = 0..4;  LX[w][l] = K[l-1] (absent for l = 0)
 *   warp totals  WT[w] = K[31]; the same Kogge-Stone over w gives WX[w] and
 *                the chunk aggregate Agg(c) = inclusive value at w = 31.
 *   look-back    c = 32k + j (32-chunk anchor intervals).  Lane lam of the
 *                look-back warp reads the fixed predecessor c-1-lam: v[lam] =
 *                Agg(c-1-lam) for lam < j, v[j] = A(k-1) (the previous
 *                interval's anchor, absent when k = 0), absent beyond.
 *                Excl(c) = PT(v[0..32)), absent for c = 0.
 *   anchor       the last chunk of each interval (j = 31) publishes
 *                A(k) = Excl(c) + Agg(c); no other chunk publishes an
 *                inclusive prefix.
 *   elements     y = (Excl(c) + WX[w]) + LX[w][l];  y = y + x_e for e = 0..,
 *                incl[cC + t] = y after adding x_e.
 *
 * Chunk size, anchor position, the shape of the fixed-order warp reduction
 * (PT over lanes) and the intra-chunk order are not fixed by the page; these
 * are the readings the library freezes.  Exclusive output is the inclusive
 * output shifted by one (excl[0] = +0.0); a reverse scan is the scan of the
 * reversed input, reversed back. */

#define NLANE 32
#define NWARP 32

/* inclusive forward scan of x[0..n) into y (y may not alias x here) */
static void FN(scan_incl_forward)(const T* x, T* y, int64_t n)
{
    const int64_t E = SCAN_E;
    const int64_t C = (int64_t)NWARP * NLANE * E;
    int64_t nchunks = (n + C - 1) / C;
    T* agg = (T*)malloc(((size_t)nchunks + 1) * sizeof(T));
    T* anchor = (T*)malloc(((size_t)nchunks / 32 + 2) * sizeof(T));
    static T LT[NWARP][NLANE], LX[NWARP][NLANE], WX[NWARP];
    for (int64_t c = 0; c < nchunks; ++c) {
        int64_t base = c * C;
        /* in-lane folds */
        for (int w = 0; w < NWARP; ++w)
            for (int l = 0; l < NLANE; ++l) {
                int64_t t0 = base + (int64_t)w * NLANE * E + (int64_t)l * E;
                T acc = (t0 < n) ? x[t0] : ABSENT;
                for (int64_t e = 1; e < E; ++e) {
                    int64_t t = t0 + e;
                    acc = acc + ((t < n) ? x[t] : ABSENT);
                }
                LT[w][l] = acc;
            }
        /* Kogge-Stone over lanes, then over warps */
        T WT[NWARP];
        for (int w = 0; w < NWARP; ++w) {
            T K[NLANE];
            for (int l = 0; l < NLANE; ++l) K[l] = LT[w][l];
            for (int r = 0; r < 5; ++r) {
                int d = 1 << r;
                T nk[NLANE];
                for (int l = 0; l < NLANE; ++l) nk[l] = (l >= d) ? K[l - d] + K[l] : K[l];
                for (int l = 0; l < NLANE; ++l) K[l] = nk[l];
            }
            for (int l = 0; l < NLANE; ++l) LX[w][l] = (l == 0) ? ABSENT : K[l - 1];
            WT[w] = K[NLANE - 1];
        }
        {
            T K[NWARP];
            for (int w = 0; w < NWARP; ++w) K[w] = WT[w];
            for (int r = 0; r < 5; ++r) {
                int d = 1 << r;
                T nk[NWARP];
                for (int w = 0; w < NWARP; ++w) nk[w] = (w >= d) ? K[w - d] + K[w] : K[w];
                for (int w = 0; w < NWARP; ++w) K[w] = nk[w];
            }
            for (int w = 0; w < NWARP; ++w) WX[w] = (w == 0) ? ABSENT : K[w - 1];
            agg[c] = K[NWARP - 1];
        }
        /* anchored look-back */
        int64_t k = c / 32, j = c % 32;
        T v[32];
        int cnt = 0;
        for (int64_t lam = 0; lam < j; ++lam) v[cnt++] = agg[c - 1 - lam];
        if (k > 0) v[cnt++] = anchor[k - 1];
        T excl = (cnt > 0) ? FN(pt)(v, cnt) : ABSENT;
        if (j == 31) anchor[k] = excl + agg[c];
        /* elements */
        for (int w = 0; w < NWARP; ++w)
            for (int l = 0; l < NLANE; ++l) {
                T yv = (excl + WX[w]) + LX[w][l];
                int64_t t0 = base + (int64_t)w * NLANE * E + (int64_t)l * E;
                for (int64_t e = 0; e < E; ++e) {
                    int64_t t = t0 + e;
                    if (t >= n) break;
                    yv = yv + x[t];
                    y[t] = yv;
                }
            }
    }
    free(anchor);
    free(agg);
}

/* flags: bit 0 = exclusive, bit 1 = reverse.  x and y may be the same array.
 * total_out (may be NULL) receives the last inclusive value in scan order
 * (+0.0 for n = 0). */
int FN(oracle_scan)(const T* x, T* y, int64_t n, int flags, T* total_out)
{
    if (n < 0 || (n > 0 && (!x || !y)) || (flags & ~3)) return 1;
    int exclusive = flags & 1, reverse = flags & 2;
    T* in = (T*)calloc((size_t)n + 1, sizeof(T));
    T* inc = (T*)malloc(((size_t)n + 1) * sizeof(T));
    for (int64_t i = 0; i < n; ++i) in[i] = reverse ? x[n - 1 - i] : x[i];
    FN(scan_incl_forward)(in, inc, n);
    if (total_out) *total_out = (n > 0) ? inc[n - 1] : (T)0.0;
    for (int64_t i = 0; i < n; ++i) {
        T o = exclusive ? ((i == 0) ? (T)0.0 : inc[i - 1]) : inc[i];
        if (reverse) y[n - 1 - i] = o; else y[i] = o;
    }
    free(inc);
    free(in);
    return 0;
}

/* ---------------------------------------------------------------------- */
/* Segmented scan: the same chunk / lane / warp / look-back structure, with
 * every '+' replaced by the segmented operator on (head flag, value) pairs,
 *   (fa, a) (+) (fb, b) = (fa | fb, fb ? b : a + b),
 * whose left operand is always the earlier part of the array.  In the
 * look-back tree higher lanes hold earlier chunks, so each node combines
 * (upper half) (+) (lower half).  Segment heads are the starts of the
 * non-empty segments given by CSR offsets.  Exclusive output is +0.0 at a
 * head and the previous inclusive value elsewhere. */

typedef struct { int f; T v; } FN(pair);

static FN(pair) FN(segop)(FN(pair) a, FN(pair) b)
{
    FN(pair) r;
    r.f = a.f | b.f;
    r.v = b.f ? b.v : a.v + b.v;
    return r;
}

static FN(pair) FN(segpt_lanes)(const FN(pair)* v, int m)
{
    if (m == 1) return v[0];
    int h = 1;
    while (h * 2 < m) h *= 2;
    FN(pair) later = FN(segpt_lanes)(v, h);         /* lanes [0, h): later chunks  */
    FN(pair) earlier = FN(segpt_lanes)(v + h, m - h); /* lanes [h, m): earlier chunks */
    return FN(segop)(earlier, later);
}

static void FN(segscan_incl_forward)(const T* x, const unsigned char* head, T* y, int64_t n)
{
    const int64_t E = SCAN_E;
    const int64_t C = (int64_t)NWARP * NLANE * E;
    int64_t nchunks = (n + C - 1) / C;
    const FN(pair) none = {0, ABSENT};
    FN(pair)* agg = (FN(pair)*)malloc(((size_t)nchunks + 1) * sizeof(FN(pair)));
    FN(pair)* anchor = (FN(pair)*)malloc(((size_t)nchunks / 32 + 2) * sizeof(FN(pair)));
    static FN(pair) LT[NWARP][NLANE], LX[NWARP][NLANE], WX[NWARP];
    for (int64_t c = 0; c < nchunks; ++c) {
        int64_t base = c * C;
        for (int w = 0; w < NWARP; ++w)
            for (int l = 0; l < NLANE; ++l) {
                int64_t t0 = base + (int64_t)w * NLANE * E + (int64_t)l * E;
                FN(pair) acc = none;
                if (t0 < n) { acc.f = head[t0]; acc.v = x[t0]; }
                for (int64_t e = 1; e < E; ++e) {
                    int64_t t = t0 + e;
                    FN(pair) el = none;
                    if (t < n) { el.f = head[t]; el.v = x[t]; }
                    acc = FN(segop)(acc, el);
                }
                LT[w][l] = acc;
            }
        FN(pair) WT[NWARP];
        for (int w = 0; w < NWARP; ++w) {
            FN(pair) K[NLANE];
            for (int l = 0; l < NLANE; ++l) K[l] = LT[w][l];
            for (int r = 0; r < 5; ++r) {
                int d = 1 << r;
                FN(pair) nk[NLANE];
                for (int l = 0; l < NLANE; ++l) nk[l] = (l >= d) ? FN(segop)(K[l - d], K[l]) : K[l];
                for (int l = 0; l < NLANE; ++l) K[l] = nk[l];
            }
            for (int l = 0; l < NLANE; ++l) LX[w][l] = (l == 0) ? none : K[l - 1];
            WT[w] = K[NLANE - 1];
        }
        {
            FN(pair) K[NWARP];
            for (int w = 0; w < NWARP; ++w) K[w] = WT[w];
            for (int r = 0; r < 5; ++r) {
                int d = 1 << r;
                FN(pair) nk[NWARP];
                for (int w = 0; w < NWARP; ++w) nk[w] = (w >= d) ? FN(segop)(K[w - d], K[w]) : K[w];
                for (int w = 0; w < NWARP; ++w) K[w] = nk[w];
            }
            for (int w = 0; w < NWARP; ++w) WX[w] = (w == 0) ? none : K[w - 1];
            agg[c] = K[NWARP - 1];
        }
        int64_t k = c / 32, j = c % 32;
        FN(pair) v[32];
        int cnt = 0;
        for (int64_t lam = 0; lam < j; ++lam) v[cnt++] = agg[c - 1 - lam];
        if (k > 0) v[cnt++] = anchor[k - 1];
        FN(pair) excl = (cnt > 0) ? FN(segpt_lanes)(v, cnt) : none;
        if (j == 31) anchor[k] = FN(segop)(excl, agg[c]);
        for (int w = 0; w < NWARP; ++w)
            for (int l = 0; l < NLANE; ++l) {
                FN(pair) yv = FN(segop)(FN(segop)(excl, WX[w]), LX[w][l]);
                int64_t t0 = base + (int64_t)w * NLANE * E + (int64_t)l * E;
                for (int64_t e = 0; e < E; ++e) {
                    int64_t t = t0 + e;
                    if (t >= n) break;
                    FN(pair) el;
                    el.f = head[t];
                    el.v = x[t];
                    yv = FN(segop)(yv, el);
                    y[t] = yv.v;
                }
            }
    }
    free(anchor);
    free(agg);
}

int FN(oracle_segmented_scan)(const T* x, T* y, int64_t n, const int64_t* offsets,
                              int64_t num_segments, int flags)
{
    if (n < 0 || num_segments < 0 || (flags & ~7)) return 1;
    if (n > 0 && (!x || !y || !offsets || num_segments < 1)) return 1;
    if (offsets) {
        if (offsets[0] != 0 || offsets[num_segments] != n) return 1;
        for (int64_t s = 0; s < num_segments; ++s)
            if (offsets[s + 1] < offsets[s]) return 1;
    }
    if (flags & 4) {
        /* Per-segment restart (flag 4): every segment is det_scan of the
         * segment alone -- its own chunk grid, look-back and anchors from the
         * segment's first element (the other reading of "segmented scans" in
         * the drjit-core pull request, "Validation"). */
        for (int64_t s = 0; s < num_segments; ++s) {
            const int64_t a = offsets[s], len = offsets[s + 1] - offsets[s];
            if (len > 0) FN(oracle_scan)(x + a, y + a, len, flags & 3, NULL);
        }
        return 0;
    }
    int exclusive = flags & 1, reverse = flags & 2;
    unsigned char* head = (unsigned char*)calloc((size_t)n + 1, 1);
    for (int64_t s = 0; s < num_segments; ++s) {
        if (offsets[s] == offsets[s + 1]) continue;
        /* forward: a segment [a, b) starts at a; reversed: at n - b */
        int64_t h = reverse ? n - offsets[s + 1] : offsets[s];
        head[h] = 1;
    }
    T* in = (T*)calloc((size_t)n + 1, sizeof(T));
    T* inc = (T*)malloc(((size_t)n + 1) * sizeof(T));
    for (int64_t i = 0; i < n; ++i) in[i] = reverse ? x[n - 1 - i] : x[i];
    FN(segscan_incl_forward)(in, head, inc, n);
    for (int64_t i = 0; i < n; ++i) {
        T o = exclusive ? (head[i] ? (T)0.0 : inc[i - 1]) : inc[i];
        if (reverse) y[n - 1 - i] = o; else y[i] = o;
    }
    free(inc);
    free(in);
    free(head);
    return 0;
}

#undef ABSENT
#undef FN
#undef CAT
#undef CAT_
