// sv_dense.cuh -- dense path: whole-row verification with a thread-block cluster per unit.
//
// A unit is (target row i, draft row i) for i <= gamma_b, or the bonus unit
// (target row gamma_b+1 alone, q := 0).  The cluster's CTAs split the
// vocabulary into contiguous column slices; every logit of the unit is read
// from HBM once (16-byte loads) and stays in registers for all the passes:
//   max            -> softmax with temperature via exp2 (one exponential per logit)
//   radix select   -> top-k (count-weighted) then top-p (mass-weighted), ties by id
//   alpha_i        =  sum_x min(p, q)
//   acceptance     u * l * q(x) < p(x)   (lenience l, 1 = the exact rule)
//   residual/bonus inverse CDF in ascending token id (hierarchical search:
//                  cluster prefix -> load group -> thread scan -> element).
// Cross-CTA values move through distributed shared memory (DSMEM) with one
// cluster barrier per exchange; partial sums are combined in fp64.
// References: "Fast Inference from Transformers via Speculative Decoding"
// review page (Algorithm 1; "Method" section on adjusted distributions) and
// "Speculative decoding: the art of guessing well", section 投机采样.
#pragma once

#include <cooperative_groups.h>

#include "sv_finalize.cuh"

namespace cg = cooperative_groups;

namespace sv {

constexpr int kXch = 32;  // doubles per exchange slot

struct DenseSmem {
    float hist[16][kDenseThreads];  // per-thread histogram columns
    float hist2[16][kDenseThreads]; // a second mass per bin (K-SEQ: the target's p beside the draft's q)
    double red[kDenseThreads / 32][kXch];
    double xch[2][kXch];
    double res[2 * kXch];
};

template <typename TIn, int R>
struct DenseCfg {
    static constexpr int NT = kDenseThreads;
    static constexpr int VEC = 16 / (int)sizeof(TIn);
    static constexpr int EPR = R * VEC;  // elements per row per thread
    static constexpr int W = NT * EPR;   // columns per CTA
};

struct Ctx {
    cg::cluster_group cl;
    int cs, crank;
    int xr;  // exchange counter (slot parity)
};

// Sum (or max) of n per-CTA values over the cluster.  `mine` lives in shared
// memory.  Afterwards res[0..n) = total, res[n..2n) = exclusive prefix over
// lower-ranked CTAs (sum only).  All threads of every CTA must call it.
__device__ __forceinline__ void cluster_combine(Ctx& c, DenseSmem& sm, const double* mine, int n, bool is_max) {
    double* slot = sm.xch[c.xr & 1];
    if (threadIdx.x < n) slot[threadIdx.x] = mine[threadIdx.x];
    c.cl.sync();
    if (threadIdx.x < n) {
        double tot = is_max ? -INFINITY : 0.0, pre = 0.0;
        for (int r = 0; r < c.cs; ++r) {
            const double v = *c.cl.map_shared_rank(&slot[threadIdx.x], r);
            if (is_max) {
                tot = fmax(tot, v);
            } else {
                if (r < c.crank) pre += v;
                tot += v;
            }
        }
        sm.res[threadIdx.x] = tot;
        sm.res[n + threadIdx.x] = pre;
    }
    __syncthreads();
    ++c.xr;
}

// Block sum of N doubles per thread; result in out[0..N) (shared), visible after return.
template <int N>
__device__ __forceinline__ void block_sum_vec(const double (&v)[N], DenseSmem& sm, double* out) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
    for (int i = 0; i < N; ++i) {
        const double s = warp_sum(v[i]);
        if (lane == 0) sm.red[wid][i] = s;
    }
    __syncthreads();
    if (threadIdx.x < N) {
        double s = 0.0;
#pragma unroll
        for (int w = 0; w < kDenseThreads / 32; ++w) s += sm.red[w][threadIdx.x];
        out[threadIdx.x] = s;
    }
    __syncthreads();
}

// The same for N floats per thread: warp sums in fp32 (32 terms), the warps'
// partials added in fp64 by N threads.
template <int N>
__device__ __forceinline__ void block_sum_vec_f(const float (&v)[N], DenseSmem& sm, double* out) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
    for (int i = 0; i < N; ++i) {
        const float s = warp_sum(v[i]);
        if (lane == 0) sm.red[wid][i] = (double)s;
    }
    __syncthreads();
    if (threadIdx.x < N) {
        double s = 0.0;
#pragma unroll
        for (int w = 0; w < kDenseThreads / 32; ++w) s += sm.red[w][threadIdx.x];
        out[threadIdx.x] = s;
    }
    __syncthreads();
}

template <int N>
__device__ __forceinline__ void block_max_vec(const double (&v)[N], DenseSmem& sm, double* out) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
    for (int i = 0; i < N; ++i) {
        double s = v[i];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s = fmax(s, __shfl_xor_sync(0xFFFFFFFFu, s, o));
        if (lane == 0) sm.red[wid][i] = s;
    }
    __syncthreads();
    if (threadIdx.x < N) {
        double s = -INFINITY;
#pragma unroll
        for (int w = 0; w < kDenseThreads / 32; ++w) s = fmax(s, sm.red[w][threadIdx.x]);
        out[threadIdx.x] = s;
    }
    __syncthreads();
}

// exclusive scan (thread order) of a double; returns the prefix, *total = block total
__device__ __forceinline__ double block_excl_scan_dbl(double v, DenseSmem& sm, double* total) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    double x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double y = __shfl_up_sync(0xFFFFFFFFu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sm.red[wid][0] = x;
    __syncthreads();
    // lane w < 8 holds warp w's total: an inclusive scan over the 8 lanes gives
    // every thread the totals before its warp and of the block
    constexpr int NW = kDenseThreads / 32;
    double wsum = lane < NW ? sm.red[lane][0] : 0.0;
#pragma unroll
    for (int o = 1; o < NW; o <<= 1) {
        const double y = __shfl_up_sync(0xFFFFFFFFu, wsum, o);
        if (lane >= o) wsum += y;
    }
    const double incl_prev = __shfl_sync(0xFFFFFFFFu, wsum, (wid + 31) & 31);
    const double tot = __shfl_sync(0xFFFFFFFFu, wsum, NW - 1);
    const double before = wid > 0 ? incl_prev : 0.0;
    __syncthreads();
    *total = tot;
    return before + (x - v);
}

template <typename TIn, int R>
__device__ __forceinline__ int col_of(const Ctx& c, int l, int j) {
    using C = DenseCfg<TIn, R>;
    return c.crank * C::W + (l * C::NT + (int)threadIdx.x) * C::VEC + j;
}

// First element, in ascending column order over the whole cluster, at which the
// running sum of the weights wgt[] passes `target` (strictly if strict, else
// reaches it); with scale_by_total the target is a fraction of the total weight.  Returns its column (the same value in every thread of every CTA),
// or -1 if every weight is zero.  *cum_incl receives the running sum including it.
template <typename TIn, int R, typename WF>
__device__ int ordered_search(Ctx& c, DenseSmem& sm, WF wgt, double target, bool strict, bool scale_by_total,
                              double* cum_incl) {
    using C = DenseCfg<TIn, R>;
    // per-thread sums of each load group (R groups of VEC consecutive columns)
    float gs[R];
#pragma unroll
    for (int l = 0; l < R; ++l) {
        float s = 0.0f;
#pragma unroll
        for (int j = 0; j < C::VEC; ++j) s += wgt(l, j);
        gs[l] = s;
    }
    double* G = sm.res + 2 * kXch - R;  // scratch tail of res, outside the exchange results
    block_sum_vec_f<R>(gs, sm, G);
    double gtot[R];
    double cta_total = 0.0;
#pragma unroll
    for (int l = 0; l < R; ++l) {
        gtot[l] = G[l];
        cta_total += gtot[l];
    }
    __shared__ double s_one[2];
    if (threadIdx.x == 0) s_one[0] = cta_total;
    __syncthreads();
    cluster_combine(c, sm, s_one, 1, false);
    const double total = sm.res[0], pre = sm.res[1];
    __syncthreads();
    if (scale_by_total) target *= total;
    // the CTA that holds the crossing, with a fallback to the last CTA with mass
    bool here = strict ? (pre <= target && target < pre + cta_total) : (pre < target && target <= pre + cta_total);
    here = here && cta_total > 0.0;
    const bool beyond = strict ? !(target < total) : !(target <= total);
    double found_col = 0.0, found_cum = 0.0;
    if (here || beyond) {
        // beyond: every CTA finds its own last positive element; the highest rank wins below
        double tl = beyond ? INFINITY : target - pre;
        int lsel = -1;
        double acc = 0.0;
#pragma unroll
        for (int l = 0; l < R; ++l) {
            if (lsel < 0 && gtot[l] > 0.0) {
                const bool in = strict ? (tl < acc + gtot[l]) : (tl <= acc + gtot[l]);
                if (in) lsel = l;
            }
            if (lsel < 0) acc += gtot[l];
        }
        if (lsel < 0) {  // rounding: last group with mass
            acc = 0.0;
#pragma unroll
            for (int l = 0; l < R; ++l)
                if (gtot[l] > 0.0) lsel = l;
#pragma unroll
            for (int l = 0; l < R; ++l)
                if (l < lsel) acc += gtot[l];
            tl = INFINITY;
        }
        const double tg = tl - acc;
        double mine = 0.0;
#pragma unroll
        for (int l = 0; l < R; ++l)
            if (l == lsel) mine = (double)gs[l];
        double tot_g;
        const double before = block_excl_scan_dbl(mine, sm, &tot_g);
        __shared__ int s_thr;
        __shared__ unsigned s_lastpos;
        if (threadIdx.x == 0) {
            s_thr = 0x7FFFFFFF;
            s_lastpos = 0u;
        }
        __syncthreads();
        const bool in_t = mine > 0.0 && (strict ? (before <= tg && tg < before + mine) : (before < tg && tg <= before + mine));
        if (in_t) atomicMin(&s_thr, (int)threadIdx.x);
        if (mine > 0.0) atomicMax(&s_lastpos, threadIdx.x + 1u);
        __syncthreads();
        int thr = s_thr;
        bool walk_all = false;
        if (thr == 0x7FFFFFFF) {
            thr = (int)s_lastpos - 1;
            walk_all = true;
        }
        if ((int)threadIdx.x == thr) {
            const double te = walk_all ? INFINITY : tg - before;
            double run = 0.0;
            int jsel = -1, jlast = -1;
            double cum_sel = 0.0, cum_last = 0.0;
#pragma unroll
            for (int l = 0; l < R; ++l) {
                if (l == lsel) {
#pragma unroll
                    for (int j = 0; j < C::VEC; ++j) {
                        const double wv = (double)wgt(l, j);
                        if (wv > 0.0) {
                            run += wv;
                            jlast = j;
                            cum_last = run;
                            if (jsel < 0 && (strict ? (te < run) : (te <= run))) {
                                jsel = j;
                                cum_sel = run;
                            }
                        }
                    }
                }
            }
            if (jsel < 0) {
                jsel = jlast;
                cum_sel = cum_last;
            }
            found_col = (double)(col_of<TIn, R>(c, lsel, jsel) + 1);
            found_cum = pre + acc + before + cum_sel;
            s_one[0] = found_col;
            s_one[1] = found_cum;
        }
        __syncthreads();
        found_col = s_one[0];
        found_cum = s_one[1];
        if (!(thr >= 0)) found_col = 0.0;
    }
    __syncthreads();
    // share: column+1 (0 = none) and the running sum; with `beyond`, the highest-rank CTA wins
    if (threadIdx.x == 0) {
        s_one[0] = (here || beyond) ? found_col : 0.0;
        s_one[1] = (here || beyond) ? found_cum : 0.0;
    }
    __syncthreads();
    double vals[2] = {s_one[0], s_one[1]};
    __syncthreads();
    double* slot = sm.xch[c.xr & 1];
    if (threadIdx.x < 2) slot[threadIdx.x] = vals[threadIdx.x];
    c.cl.sync();
    if (threadIdx.x == 0) {
        double col = 0.0, cum = 0.0;
        for (int r = 0; r < c.cs; ++r) {
            const double cc = *c.cl.map_shared_rank(&slot[0], r);
            if (cc > 0.0) {
                if (col == 0.0 || beyond) {  // strict hit is unique; fallback takes the last
                    col = cc;
                    cum = *c.cl.map_shared_rank(&slot[1], r);
                }
            }
        }
        sm.res[0] = col;
        sm.res[1] = cum;
    }
    __syncthreads();
    ++c.xr;
    const int col = (int)sm.res[0] - 1;
    *cum_incl = sm.res[1];
    __syncthreads();
    return col;
}

// Keep the shortest prefix of the (e desc, column asc) order whose weight
// (1 per element if !mass, else e) reaches `target`; zero e elsewhere.
// Keys are the bit patterns of the non-negative floats e (monotone).
template <typename TIn, int R>
__device__ void select_keep(Ctx& c, DenseSmem& sm, float (&e)[DenseCfg<TIn, R>::EPR], int V, bool mass,
                            double target) {
    using C = DenseCfg<TIn, R>;
    const int t = threadIdx.x;
    uint32_t prefix = 0u;
    double above = 0.0;
    bool keep_all = false;
    for (int d = 7; d >= 0; --d) {
        const int sh = 4 * d;
#pragma unroll
        for (int bin = 0; bin < 16; ++bin) sm.hist[bin][t] = 0.0f;
#pragma unroll
        for (int l = 0; l < R; ++l) {
#pragma unroll
            for (int j = 0; j < C::VEC; ++j) {
                const int i = l * C::VEC + j;
                if (col_of<TIn, R>(c, l, j) < V) {
                    const uint32_t key = __float_as_uint(e[i]);
                    const bool match = (d == 7) || ((key >> (sh + 4)) == (prefix >> (sh + 4)));
                    if (match) sm.hist[(key >> sh) & 15u][t] += mass ? e[i] : 1.0f;
                }
            }
        }
        __syncthreads();
        // block-reduce the 16 bins: thread t sums 16 columns of bin (t & 15)
        {
            const int bin = t & 15, part = t >> 4;
            float s = 0.0f;
#pragma unroll
            for (int i = 0; i < 16; ++i) s += sm.hist[bin][part * 16 + i];
            s += __shfl_xor_sync(0xFFFFFFFFu, s, 16);
            const int wid = t >> 5, lane = t & 31;
            if (lane < 16) sm.red[wid][lane] = (double)s;
        }
        __syncthreads();
        __shared__ double s_bins[16];
        if (t < 16) {  // read back by this same thread in the exchange below
            double s = 0.0;
#pragma unroll
            for (int w = 0; w < kDenseThreads / 32; ++w) s += sm.red[w][t];
            s_bins[t] = s;
        }
        cluster_combine(c, sm, s_bins, 16, false);
        // the digit: one thread walks the 16 bins (an fp64 chain), the block reads it
        __shared__ double s_above;
        __shared__ int s_dsel, s_keep_all;
        if (t == 0) {
            double acc = above;
            int dsel = -1, lowest = -1, all = 0;
            for (int bin = 15; bin >= 0; --bin) {
                const double g = sm.res[bin];
                if (g > 0.0) lowest = bin;
                if (dsel < 0 && g > 0.0 && acc + g >= target) dsel = bin;
                if (dsel < 0) acc += g;
            }
            if (dsel < 0) {  // the weight never reaches the target (rounding): keep everything
                all = 1;
                dsel = (lowest < 0) ? 0 : lowest;
                acc = above;
                for (int bin = 15; bin > dsel; --bin) acc += sm.res[bin];
            }
            s_above = acc;
            s_dsel = dsel;
            s_keep_all = all;
        }
        __syncthreads();
        above = s_above;
        keep_all = s_keep_all != 0;
        prefix |= (uint32_t)s_dsel << sh;
        if (keep_all) break;
    }
    if (keep_all) return;
    // ties at the boundary key, in ascending column order
    const uint32_t kappa = prefix;
    auto wt = [&](int l, int j) -> float {
        const int i = l * C::VEC + j;
        const bool tie = col_of<TIn, R>(c, l, j) < V && __float_as_uint(e[i]) == kappa;
        return tie ? (mass ? e[i] : 1.0f) : 0.0f;
    };
    double cum;
    const int cstar = ordered_search<TIn, R>(c, sm, wt, target - above, false, false, &cum);
#pragma unroll
    for (int l = 0; l < R; ++l)
#pragma unroll
        for (int j = 0; j < C::VEC; ++j) {
            const int i = l * C::VEC + j;
            const int col = col_of<TIn, R>(c, l, j);
            const uint32_t key = __float_as_uint(e[i]);
            const bool keep = col < V && (key > kappa || (key == kappa && col <= cstar));
            if (!keep) e[i] = 0.0f;
        }
}

template <typename TIn, int R, bool VECTOR>
__device__ __forceinline__ void load_row(const TIn* row, const Ctx& c, int V, float (&x)[DenseCfg<TIn, R>::EPR],
                                         bool& bad) {
    using C = DenseCfg<TIn, R>;
#pragma unroll
    for (int l = 0; l < R; ++l) {
        const int col = col_of<TIn, R>(c, l, 0);
        uint32_t wv[4] = {0u, 0u, 0u, 0u};
        if (VECTOR) {
            if (col < V) {
                const uint4 v = ld_stream16(row + col);
                wv[0] = v.x;
                wv[1] = v.y;
                wv[2] = v.z;
                wv[3] = v.w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < C::VEC; ++j)
                if (col + j < V) {
                    const uint32_t bits = (sizeof(TIn) == 4) ? __ldg((const unsigned int*)row + col + j)
                                                             : (uint32_t)__ldg((const unsigned short*)row + col + j);
                    wv[j / (4 / (int)sizeof(TIn))] |= bits << ((sizeof(TIn) == 2 && (j & 1)) ? 16 : 0);
                }
        }
#pragma unroll
        for (int j = 0; j < C::VEC; ++j) {
            uint32_t bits;
            if (sizeof(TIn) == 4) {
                bits = wv[j];
            } else {
                const uint32_t h = (j & 1) ? (wv[j >> 1] >> 16) : (wv[j >> 1] & 0xFFFFu);
                bad |= (col + j < V) && bad16(h);
                bits = h << 16;
            }
            if (sizeof(TIn) == 4) bad |= (col + j < V) && bad32(bits);
            x[l * C::VEC + j] = (col + j < V) ? __uint_as_float(bits) : -INFINITY;
        }
    }
}

// K-SEQ verification of one position with k candidates ("SpecTr: Fast
// Speculative Decoding via Optimal Transport" page, section K-SEQ, eqs. (4)-(7)
// and the residual distribution; the page names the draft p and the target q,
// here p is the target and q the draft).  p, q: the unit's normalised rows held
// by this cluster.  With m(x) = min(q(x), p(x) / rho) and beta(rho) = sum_x m(x):
//   rho* solves 1 - (1 - beta)^k = rho beta on [1, k] (the left side minus the right,
//     f, does not increase with rho);
//   candidate i (in the given order) is accepted iff u_i rho* q(X_i) < p(X_i);
//   if none is, the token is drawn from p - A, A = (P_A / beta) m(x) at rho*,
//     P_A = 1 - (1 - beta)^k, by the inverse CDF in ascending token id.
// rho*: beta(rho) = Q(rho) + P(rho) / rho with Q the draft mass of the tokens whose
// ratio r = p / q is at least rho and P the target mass of the others (tokens with
// p = 0 or q = 0 add nothing).  A radix descent over the float bits of rho finds the
// largest float rho_lo with f(rho_lo) > 0, four bits per round, f being evaluated
// in fp64 at the 16 digit boundaries from a cluster histogram of the q and p mass
// of the ratio keys in the current range; inside (rho_lo, next float) no ratio
// lies, so Q and P are constants there and f, affine there to within rounding,
// is zero at the interpolation of its values at the two ends.
template <typename TIn, int R>
__device__ void kseq_unit(const Args& a, Ctx& c, DenseSmem& sm, double* s_vals, const float (&p)[DenseCfg<TIn, R>::EPR],
                          const float (&q)[DenseCfg<TIn, R>::EPR], int b, int k, int V) {
    using C = DenseCfg<TIn, R>;
    const int t = threadIdx.x;
    const double kd = (double)k;
    // rho^k f(rho) = rho^k (1 - rho Q - P) - (rho (1 - Q) - P)^k for fixed Q, P (rho beta =
    // rho Q + P and 1 - beta = (rho (1 - Q) - P) / rho): the sign of f without a
    // division; k <= 13 products on each side
    auto fk = [&](double rho, double Q, double P) -> double {
        const double lhs = 1.0 - rho * Q - P, base = rho * (1.0 - Q) - P;
        double rk = 1.0, bk = 1.0;
        for (int i = 0; i < k; ++i) {
            rk *= rho;
            bk *= base;
        }
        return rk * lhs - bk;
    };
    // ---- the radix descent.  Per round: each thread bins its own elements into
    // its column of the (q, p) histograms; 8 threads per column sum them
    // (compensated fp32); 32 threads add the 8 partials in fp64; the cluster sums
    // them; warp 0 evaluates f at the 16 digit boundaries (16-lane scans) and
    // carries Q (q mass above the range) and P (p mass below it) in registers.
    // The ratio key is the float bits of p / q by the fast reciprocal: the same
    // key in every round, so the histograms stay consistent; a ratio within two
    // ulps of rho* changes beta by that fraction of the token's own mass.
    uint32_t prefix = 0u;
    double Qhi = 0.0, Plo = 0.0, Pfin = 0.0;  // meaningful in warp 0
    __shared__ int s_sel;
    for (int d = 7; d >= 0; --d) {
        const int sh = 4 * d;
#pragma unroll
        for (int bin = 0; bin < 16; ++bin) {
            sm.hist[bin][t] = 0.0f;
            sm.hist2[bin][t] = 0.0f;
        }
#pragma unroll
        for (int l = 0; l < R; ++l)
#pragma unroll
            for (int j = 0; j < C::VEC; ++j) {
                const int i = l * C::VEC + j;
                if (col_of<TIn, R>(c, l, j) < V && p[i] > 0.0f && q[i] > 0.0f) {
                    const uint32_t key = __float_as_uint(__fdividef(p[i], q[i]));
                    if (d == 7 || (key >> (sh + 4)) == (prefix >> (sh + 4))) {
                        sm.hist[(key >> sh) & 15u][t] += q[i];
                        sm.hist2[(key >> sh) & 15u][t] += p[i];
                    }
                }
            }
        __syncthreads();
        {  // partial sums of the 32 (bin, mass) columns: 8 threads per column, Kahan in fp32
            const int col = t & 31, part = t >> 5;
            const float* h = (col < 16) ? &sm.hist[col][0] : &sm.hist2[col - 16][0];
            float sum = 0.0f, comp = 0.0f;
#pragma unroll 8
            for (int i = 0; i < kDenseThreads / 8; ++i) {
                const float y = h[part * (kDenseThreads / 8) + i] - comp;
                const float tt = sum + y;
                comp = (tt - sum) - y;
                sum = tt;
            }
            sm.red[part][col] = (double)sum - (double)comp;
        }
        __syncthreads();
        if (t < 32) {
            double sum = 0.0;
#pragma unroll
            for (int w = 0; w < 8; ++w) sum += sm.red[w][t];
            s_vals[t] = sum;  // read back by this same thread in the exchange below
        }
        cluster_combine(c, sm, s_vals, 32, false);
        if (t < 32) {
            // digit t of this round: is f > 0 at the start of its range?  (rho < 1: yes,
            // f(1) >= 0 and rho* >= 1; rho > k: no; sign-bit keys are not ratios)
            // Q_t = Qhi + sum_{j >= t} q_j and P_t = Plo + sum_{j < t} p_j by 16-lane scans
            double qs = t < 16 ? sm.res[15 - t] : 0.0, ps = t < 16 ? sm.res[16 + t] : 0.0;
#pragma unroll
            for (int o = 1; o < 16; o <<= 1) {
                const double qy = __shfl_up_sync(0xFFFFFFFFu, qs, o), py = __shfl_up_sync(0xFFFFFFFFu, ps, o);
                if ((t & 15) >= o) {
                    qs += qy;
                    ps += py;
                }
            }
            // lane t: qs = sum_{j >= 15 - t} q_j, ps = sum_{j <= t} p_j (lanes 16..31: 0)
            const double q_ge = __shfl_sync(0xFFFFFFFFu, qs, (15 - t) & 31);  // sum_{j >= t} q_j
            const double p_prev = __shfl_sync(0xFFFFFFFFu, ps, (t + 31) & 31);
            const double p_lt = t > 0 ? p_prev : 0.0;  // sum_{j < t} p_j
            bool pos = false;
            if (t < 16 && !(d == 7 && t >= 8)) {
                const float rho_f = __uint_as_float(prefix | ((uint32_t)t << sh));
                const double rho = (double)rho_f;
                if (rho < 1.0) {
                    pos = true;
                } else if (rho <= kd) {
                    pos = fk(rho, Qhi + q_ge, Plo + p_lt) > 0.0;
                }
            }
            const unsigned m = __ballot_sync(0xFFFFFFFFu, pos);
            const int sel = m ? 31 - __clz(m) : 0;  // f does not increase: the largest such digit
            // carry: the q mass of the digits above sel, the p mass of those below it; the
            // keys equal to the final prefix (the last round's digit) lie below every rho
            // inside (rho_lo, next float): their p mass joins P
            const double q_above = __shfl_sync(0xFFFFFFFFu, q_ge, (sel + 1) & 31);  // lane 16: 0
            const double p_below = __shfl_sync(0xFFFFFFFFu, p_lt, sel);
            const double p_upto = __shfl_sync(0xFFFFFFFFu, ps, sel);
            Pfin = Plo + p_upto;
            Qhi += q_above;
            Plo += p_below;
            if (t == 0) s_sel = sel;
        }
        __syncthreads();
        prefix |= (uint32_t)s_sel << sh;
    }
    const double Q = Qhi, P = Pfin;  // thread 0's values are the ones used below
    __shared__ double s_rho, s_beta;
    __shared__ int s_tok, s_idx;
    if (t == 0) {
        // inside [lo, hi] (at most one float step wide, relative 1.2e-7) f is affine to
        // within rounding: the root is the interpolation of its two ends
        double lo = fmax(1.0, (double)__uint_as_float(prefix));
        double hi = fmin(kd, (double)__uint_as_float(prefix + 1u));
        double rho = hi;
        if (lo < hi) {
            auto f = [&](double r) {
                const double beta = Q + (P > 0.0 ? P / r : 0.0);
                double pw = 1.0;
                for (int i = 0; i < k; ++i) pw *= (1.0 - beta);
                return 1.0 - pw - r * beta;
            };
            const double flo = f(lo), fhi = f(hi);
            if (flo > 0.0 && fhi < 0.0) rho = lo + (hi - lo) * (flo / (flo - fhi));
            else rho = flo > 0.0 ? hi : lo;
        }
        s_rho = rho;
        s_beta = Q + (P > 0.0 ? P / rho : 0.0);
    }
    __syncthreads();
    const double rho = s_rho, beta = s_beta;
    // ---- the candidates' probabilities: each column is held by one thread of the
    // cluster, which writes them to its CTA's slots; the cluster sum collects them
    __shared__ int s_cand[SV_MAX_KSEQ];
    if (t < SV_MAX_KSEQ) s_cand[t] = t < k ? a.draft_tokens[(size_t)b * a.G + t] : -1;
    if (t < 2 * SV_MAX_KSEQ) s_vals[t] = 0.0;
    __syncthreads();
#pragma unroll
    for (int l = 0; l < R; ++l)
#pragma unroll
        for (int j = 0; j < C::VEC; ++j) {
            const int col = col_of<TIn, R>(c, l, j);
            if (col >= V) continue;
            for (int i = 0; i < k; ++i)
                if (s_cand[i] == col) {
                    s_vals[2 * i] = (double)p[l * C::VEC + j];
                    s_vals[2 * i + 1] = (double)q[l * C::VEC + j];
                }
        }
    __syncthreads();
    cluster_combine(c, sm, s_vals, 2 * SV_MAX_KSEQ, false);
    if (t == 0) {
        int idx = -1;
        for (int i = 0; i < k && idx < 0; ++i) {
            const double u = uniform01(a.seed, (uint32_t)b, 1u, 3u + (uint32_t)i);
            if (u * rho * sm.res[2 * i + 1] < sm.res[2 * i]) idx = i;
        }
        s_idx = idx;
        s_tok = idx >= 0 ? s_cand[idx] : -1;
    }
    __syncthreads();
    int token = s_tok;
    const int idx = s_idx;
    if (idx < 0) {
        // ---- the residual p - A at rho*, by the inverse CDF in ascending id
        const double PA = beta > 0.0 ? 1.0 - [&] {
            double pw = 1.0;
            for (int i = 0; i < k; ++i) pw *= (1.0 - beta);
            return pw;
        }() : 0.0;
        const float As = beta > 0.0 ? (float)(PA / beta) : 0.0f;
        const float inv_rho = (float)(1.0 / rho);
        auto resid = [&](int l, int j) -> float {
            const int i = l * C::VEC + j;
            return fmaxf(p[i] - As * fminf(q[i], p[i] * inv_rho), 0.0f);
        };
        float rs = 0.0f;
#pragma unroll
        for (int l = 0; l < R; ++l)
#pragma unroll
            for (int j = 0; j < C::VEC; ++j) rs += resid(l, j);
        double z1[1] = {(double)rs};
        block_sum_vec<1>(z1, sm, s_vals);
        cluster_combine(c, sm, s_vals, 1, false);
        const double Z = sm.res[0];
        __syncthreads();
        const double ur = uniform01(a.seed, (uint32_t)b, 1u, 1u);
        double cum;
        if (Z > 0.0)
            token = ordered_search<TIn, R>(c, sm, resid, ur, true, true, &cum);
        else  // no residual mass (P_A = 1 up to rounding): fall back to p
            token = ordered_search<TIn, R>(
                c, sm, [&](int l, int j) -> float { return p[l * C::VEC + j]; }, ur, true, true, &cum);
    }
    if (c.crank == 0 && t == 0) {
        a.out_tokens[b] = token;
        a.accepted_len[b] = idx;
        if (a.row_status) a.row_status[b] = 0u;
    }
}

template <typename TIn, int R, bool VECTOR>
__global__ void __launch_bounds__(kDenseThreads, 1) dense_kernel(Args a) {
    using C = DenseCfg<TIn, R>;
    __shared__ DenseSmem sm;
    __shared__ double s_vals[kXch];
    Ctx c{cg::this_cluster(), 0, 0, 0};
    c.cs = (int)c.cl.num_blocks();
    c.crank = (int)c.cl.block_rank();
    const int t = threadIdx.x;
    const int V = a.V, G = a.G;
    // No unit from the plan and no whole-row unit that could be handed over (only
    // nucleus units can be): leave at once, without waiting for the kernels before
    // this one (both counts are the plan's, final and visible here, as in free_kernel)
    if (a.counts[kCntDenseUnits] == 0u && a.counts[kCntFreeNucUnits] == 0u) return;
    grid_dependency_wait();  // the previous kernels of the call (the plan's lists, the handovers)
    const uint32_t n_units = a.counts[kCntDenseUnits];
    if (n_units == 0) return;  // nothing for any cluster: no shared memory is ever shared
    // a wait of an earlier kernel gave up: the whole-row tail kernel has then
    // already finished (as failed) every unit that kernel handed over here
    const bool failed = a.counts[kCntError] != 0u;
    const uint32_t cid = blockIdx.x / (uint32_t)c.cs, ncl = gridDim.x / (uint32_t)c.cs;

    for (uint32_t w = cid; w < n_units; w += ncl) {
        const uint32_t item = a.dense_units[w];
        const int b = (int)(item >> 8), u = (int)(item & 0xFFu);
        const SeqInfo si = a.seq[b];
        if (failed && si.mode == kModeFree) continue;  // uniform over the cluster: every CTA skips it
        const bool has_draft = u < si.gamma;
        const bool pair = has_draft && !a.gumbel;  // the draft row is read (not by shared noise)
        const float Lb = si.L;
        // K-SEQ rows are [B, V] (one position per row); otherwise target [B, G+1, V], draft [B, G, V]
        const TIn* trow = (const TIn*)a.target + (a.kseq ? (size_t)b : (size_t)b * (G + 1) + u) * (size_t)V;
        const TIn* drow = (const TIn*)a.draft + (a.kseq ? (size_t)b : (size_t)b * G + u) * (size_t)V;

        float xt[C::EPR], xd[C::EPR];
        bool bad = false;
        load_row<TIn, R, VECTOR>(trow, c, V, xt, bad);
        if (pair) {
            load_row<TIn, R, VECTOR>(drow, c, V, xd, bad);
        } else {
#pragma unroll
            for (int i = 0; i < C::EPR; ++i) xd[i] = -INFINITY;
        }

        // ---- maxima (and the non-finite flag) over the cluster
        {
            float mt = -INFINITY, md = -INFINITY;
#pragma unroll
            for (int i = 0; i < C::EPR; ++i) {
                mt = fmaxf(mt, xt[i]);
                md = fmaxf(md, xd[i]);
            }
            double v3[3] = {(double)mt, (double)md, bad ? 1.0 : 0.0};
            block_max_vec<3>(v3, sm, s_vals);
            cluster_combine(c, sm, s_vals, 3, true);
        }
        const float Mt = (float)sm.res[0], Md = (float)sm.res[1];
        const bool nonfinite = sm.res[2] > 0.0 || !(Mt > -INFINITY) || (pair && !(Md > -INFINITY));
        __syncthreads();
        if (nonfinite) {
            if (c.crank == 0) {
                if (a.kseq) {
                    if (t == 0) {
                        a.out_tokens[b] = -1;
                        a.accepted_len[b] = -1;
                        if (a.row_status) a.row_status[b] = SV_ROW_NONFINITE;
                    }
                } else {
                    if (t == 0) atomicOr(&a.seq_status[b], SV_ROW_NONFINITE);
                    unit_finished(a, b);
                }
            }
            continue;
        }

        // ---- exponentials: e = 2^((x - M) log2(e) / T); greedy: indicator of the maximum
        const bool greedy = (si.T == 0.0f);
        const float cscale = greedy ? 0.0f : (float)(1.4426950408889634 / (double)si.T);
#pragma unroll
        for (int i = 0; i < C::EPR; ++i) {
            if (greedy) {
                xt[i] = (xt[i] == Mt) ? 1.0f : 0.0f;
                xd[i] = (pair && xd[i] == Md) ? 1.0f : 0.0f;
            } else {
                xt[i] = exp2f(fmaf(xt[i], cscale, -Mt * cscale));
                xd[i] = pair ? exp2f(fmaf(xd[i], cscale, -Md * cscale)) : 0.0f;
            }
        }

        // ---- filters (greedy: keep the lowest-id maximum only)
        const int kf = greedy ? 1 : si.k;
        const float Pf = greedy ? 1.0f : si.P;
        if (kf > 0) {
            select_keep<TIn, R>(c, sm, xt, V, false, (double)kf);
            if (pair) select_keep<TIn, R>(c, sm, xd, V, false, (double)kf);
        }
        if (Pf < 1.0f) {
            double sums[2] = {0.0, 0.0};
            float st = 0.0f, sd = 0.0f;
#pragma unroll
            for (int i = 0; i < C::EPR; ++i) {
                st += xt[i];
                sd += xd[i];
            }
            sums[0] = st;
            sums[1] = sd;
            block_sum_vec<2>(sums, sm, s_vals);
            cluster_combine(c, sm, s_vals, 2, false);
            const double St = sm.res[0], Sd = sm.res[1];
            __syncthreads();
            select_keep<TIn, R>(c, sm, xt, V, true, (double)Pf * St);
            if (pair) select_keep<TIn, R>(c, sm, xd, V, true, (double)Pf * Sd);
        }

        if (a.gumbel) {
            // ---- shared noise ("Speculative decoding: the art of guessing well", section
            // 共享噪声的采样): the target's token is the argmax over the kept tokens of
            // log p + g; log of the kept weight 2^((x - M) log2(e) / T) is (x - M) / T, the
            // renormalisation being one constant; ties go to the lower id; greedy: the
            // one kept token
            const uint32_t k0 = (uint32_t)a.seed, k1 = (uint32_t)(a.seed >> 32);
            float bs = -INFINITY;
            int bid = 0x7FFFFFFF;
#pragma unroll
            for (int l = 0; l < R; ++l) {
                const int col0 = col_of<TIn, R>(c, l, 0);  // a multiple of 4
#pragma unroll
                for (int h = 0; h < C::VEC / 4; ++h) {
                    uint4 wq = make_uint4(0u, 0u, 0u, 0u);
                    if (!greedy && col0 + 4 * h < V)
                        wq = philox4((uint32_t)b, (uint32_t)(u + 1), 2u, (uint32_t)(col0 >> 2) + h, k0, k1);
                    const uint32_t ws4[4] = {wq.x, wq.y, wq.z, wq.w};
#pragma unroll
                    for (int j4 = 0; j4 < 4; ++j4) {
                        const int j = 4 * h + j4, col = col0 + j;
                        const float e = xt[l * C::VEC + j];
                        if (col < V && e > 0.0f) {
                            const float sc =
                                greedy ? 0.0f : fmaf(__log2f(e), 0.693147180559945309f, gumbel_of_word(ws4[j4]));
                            if (sc > bs || (sc == bs && col < bid)) {
                                bs = sc;
                                bid = col;
                            }
                        }
                    }
                }
            }
            // over the cluster: the largest score, then the lowest id holding it
            double v1[1] = {(double)bs};
            block_max_vec<1>(v1, sm, s_vals);
            cluster_combine(c, sm, s_vals, 1, true);
            const float top = (float)sm.res[0];
            __syncthreads();
            double v2[1] = {bs == top ? -(double)bid : -INFINITY};
            block_max_vec<1>(v2, sm, s_vals);
            cluster_combine(c, sm, s_vals, 1, true);
            const int token = (int)(-sm.res[0]);
            __syncthreads();
            if (c.crank == 0) {
                if (t == 0) {
                    if (has_draft) {
                        const int acc = a.draft_tokens[(size_t)b * G + u] == token ? 1 : 0;
                        a.unit_acc[(size_t)b * G + u] = acc;
                        if (a.pos_accept) a.pos_accept[(size_t)b * G + u] = acc;
                    }
                    a.unit_tok[(size_t)b * (G + 1) + u] = token;
                    if (a.pos_token) a.pos_token[(size_t)b * (G + 1) + u] = token;
                }
                unit_finished(a, b);
            }
            continue;
        }

        // ---- normalisers of the kept mass
        double St, Sd;
        {
            double sums[2];
            float st = 0.0f, sd = 0.0f;
#pragma unroll
            for (int i = 0; i < C::EPR; ++i) {
                st += xt[i];
                sd += xd[i];
            }
            sums[0] = st;
            sums[1] = sd;
            block_sum_vec<2>(sums, sm, s_vals);
            cluster_combine(c, sm, s_vals, 2, false);
            St = sm.res[0];
            Sd = sm.res[1];
            __syncthreads();
        }
        const float inv_t = (float)(1.0 / St);
        const float inv_d = pair ? (float)(1.0 / Sd) : 0.0f;
#pragma unroll
        for (int i = 0; i < C::EPR; ++i) {
            xt[i] *= inv_t;  // p
            xd[i] *= inv_d;  // q
        }

        // ---- debug copies of the normalised rows
        if (a.p_out || a.q_out) {
#pragma unroll
            for (int l = 0; l < R; ++l)
#pragma unroll
                for (int j = 0; j < C::VEC; ++j) {
                    const int col = col_of<TIn, R>(c, l, j);
                    if (col < V) {
                        if (a.p_out) a.p_out[((size_t)b * (G + 1) + u) * V + col] = xt[l * C::VEC + j];
                        if (a.q_out && pair) a.q_out[((size_t)b * G + u) * V + col] = xd[l * C::VEC + j];
                    }
                }
        }

        if (a.kseq) {
            kseq_unit<TIn, R>(a, c, sm, s_vals, xt, xd, b, si.gamma, V);
            continue;
        }

        // ---- alpha, acceptance gather; the residual weights replace q in place
        const int x_tok = pair ? a.draft_tokens[(size_t)b * G + u] : -1;
        const float invl = lenience_inv(Lb);  // alpha under lenience: sum_x min(q, p / l)
        double part[4] = {0.0, 0.0, 0.0, 0.0};
        {
            float al = 0.0f, rs = 0.0f;
#pragma unroll
            for (int l = 0; l < R; ++l)
#pragma unroll
                for (int j = 0; j < C::VEC; ++j) {
                    const int i = l * C::VEC + j;
                    const float p = xt[i], q = xd[i];
                    al += accept_mass(p, q, invl);
                    if (col_of<TIn, R>(c, l, j) == x_tok) {
                        part[1] = (double)p;
                        part[2] = (double)q;
                    }
                    xd[i] = pair ? fmaxf(p - q, 0.0f) : p;  // bonus: q_{gamma+1} := 0
                    rs += xd[i];
                }
            part[0] = (double)al;
            part[3] = (double)rs;
        }
        block_sum_vec<4>(part, sm, s_vals);
        cluster_combine(c, sm, s_vals, 4, false);
        const double alpha = sm.res[0], px = sm.res[1], qx = sm.res[2];
        const double Z = sm.res[3];
        __syncthreads();
        if (!(Z > 0.0)) {  // p <= q everywhere: the draw falls back to p
#pragma unroll
            for (int i = 0; i < C::EPR; ++i) xd[i] = xt[i];
        }
        const double ua = uniform01(a.seed, (uint32_t)b, (uint32_t)(u + 1), 0u);
        const double ur = uniform01(a.seed, (uint32_t)b, (uint32_t)(u + 1), 1u);
        double cum;
        // v = u * Z, with Z the search's own hierarchical total, so that v < Z exactly
        const int token = ordered_search<TIn, R>(
            c, sm, [&](int l, int j) -> float { return xd[l * C::VEC + j]; }, ur, true, true, &cum);
        const int accept = pair ? (lenient_accept(ua, Lb, qx, px) ? 1 : 0) : 0;

        if (c.crank == 0) {
            if (t == 0) {
                if (pair) {
                    a.alpha[(size_t)b * G + u] = (float)alpha;
                    a.unit_acc[(size_t)b * G + u] = accept;
                    if (a.pos_accept) a.pos_accept[(size_t)b * G + u] = accept;
                }
                a.unit_tok[(size_t)b * (G + 1) + u] = token;
                if (a.pos_token) a.pos_token[(size_t)b * (G + 1) + u] = token;
            }
            unit_finished(a, b);
        }
    }
    // no CTA may leave while a peer can still read its shared memory
    c.cl.sync();
}

// Vocabulary split: load groups per thread R and cluster size cs (R * cs is
// about V / 2048 for bf16, V / 1024 for fp32).  A unit's time is mostly its
// rounds of cluster-wide exchanges, so the smallest R (the shortest per-thread
// loops) serves a batch whose units fit the GPU's clusters at once; a batch with
// more units than that takes the largest R, whose smaller clusters run more
// units side by side (the batch's unit count is an upper bound: the plan picks
// the units on the device).
template <typename TIn>
inline bool dense_shape(int V, long long units, int sms, int* R, int* cs) {
    const int vec = 16 / (int)sizeof(TIn);
    const int rmax = sizeof(TIn) == 2 ? 8 : 16;
    int n = 0, rs[8], cl[8];
    for (int r = 1; r <= rmax; r <<= 1) {
        const int w = kDenseThreads * r * vec;
        const int c = (V + w - 1) / w;
        if (c <= 8 || (r == rmax && c <= 16)) {
            rs[n] = r;
            cl[n] = c;
            ++n;
        }
    }
    if (n == 0) return false;
    int pick = 0;
    if (units > (long long)(sms / cl[0])) pick = n - 1;
    *R = rs[pick];
    *cs = cl[pick];
    return true;
}

// Persistent launch: as many clusters as fit on the GPU at once, each walking
// the dense unit list.
template <typename TIn, int R, bool VECTOR>
cudaError_t launch_dense_cluster(const Args& a, int cs, int sms, cudaStream_t s) {
    auto k = dense_kernel<TIn, R, VECTOR>;
    static const bool attr_ok = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess;
    (void)attr_ok;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(kDenseThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3((unsigned)cs);
    // clusters of size cs resident at once (queried on the first launch of each size)
    static int cached[17] = {};
    if (cs < 1 || cs > 16) return cudaErrorInvalidValue;
    int clusters = cached[cs];
    if (clusters < 1) {
        if (cudaOccupancyMaxActiveClusters(&clusters, k, &cfg) != cudaSuccess || clusters < 1) {
            (void)cudaGetLastError();
            clusters = sms / cs > 0 ? sms / cs : 1;
        }
        cached[cs] = clusters;
    }
    const long long upper = (long long)a.B * (a.G + 1);
    long long n = clusters;
    if (n > upper) n = upper;
    if (n < 1) n = 1;
    const cudaError_t e = launch_pdl(k, dim3((unsigned)(n * cs)), dim3(kDenseThreads), 0, s, a, attr, 1);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace sv
