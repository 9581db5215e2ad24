// Temperature sampling of the draft-and-verify round (T > 0): speculative
// rejection sampling, "DFlash: Why a Diffusion Drafter Can Accelerate an
// Autoregressive Model" §4.2 (eq. 6-8) and Algorithm 1 (steps 2-3, 7-8, 10);
// "DFlash: Block Diffusion for Flash Speculative Decoding", Paper vs code
// "Sampling rule" (top-p and top-k apply to both distributions).
//
// Laws are softmax(logits / T) of fp32 logit rows, filtered by top-k / top-p:
// q from the draft head's rows 1..B-1, p from the verify head's rows 0..B-1
// (p_j decides the proposal at block row j + 1).  Tokens rank by logit, highest
// first, equal logits in increasing id; top-k keeps the first k, top-p then
// keeps each token whose top-k mass ranked before it is below p.  A filtered
// law is stored as (max, kept sum, threshold key, threshold id): token z is
// kept when its (key, id) ranks at or above the threshold.  Every draw is an
// inverse-CDF lookup of a caller-supplied uniform u in [0, 1): the lowest token
// z whose cumulative weight exceeds u * total.
//
// One thread-block cluster handles one law row (statistics, threshold, draw) or
// one sequence (acceptance and the emitted token): CTA r of the cluster owns
// the r-th contiguous chunk of the vocabulary.  The law kernels stage their
// chunk in shared memory once (one pass over the logits in HBM / L2); every
// later pass (the radix selections of the thresholds, the kept sum, the draw)
// reads shared memory.  Partial results are combined across the cluster
// through distributed shared memory in CTA order, so every sum has one fixed
// order and every selection is exact (integer histograms).
#include <cooperative_groups.h>
#include <math.h>

#include "launch.h"
#include "loss.h"

namespace cg = cooperative_groups;

namespace dfl {

namespace {

constexpr int SNT = 1024;  // threads per sampling CTA

// Row statistics of softmax(l / T): m = max l, s = sum exp((l - m) / T).
__device__ float block_max_f(float v, float* red) {
    v = warp_max(v);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    if (l == 0) red[w] = v;
    __syncthreads();
    if (w == 0) {
        v = l < (int)(blockDim.x >> 5) ? red[l] : -INFINITY;
        v = warp_max(v);
        if (l == 0) red[0] = v;
    }
    __syncthreads();
    v = red[0];
    __syncthreads();
    return v;
}

__device__ float block_sum_f(float v, float* red) {
    v = warp_sum(v);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    if (l == 0) red[w] = v;
    __syncthreads();
    if (w == 0) {
        v = l < (int)(blockDim.x >> 5) ? red[l] : 0.f;
        v = warp_sum(v);
        if (l == 0) red[0] = v;
    }
    __syncthreads();
    v = red[0];
    __syncthreads();
    return v;
}

// Sum of w(z) over z = first, first + stride, ... < end with eight independent
// partial sums (eight loads in flight per thread), combined in a fixed order.
template <class W>
__device__ __forceinline__ float strided_sum(const W& w, int first, int end, int stride) {
    float p[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    int z = first;
    for (; z + 7 * stride < end; z += 8 * stride) {
#pragma unroll
        for (int k = 0; k < 8; ++k) p[k] += w(z + k * stride);
    }
#pragma unroll
    for (int k = 0; k < 8; ++k)  // fewer than 8 left
        if (z + k * stride < end) p[k] += w(z + k * stride);
    return ((p[0] + p[1]) + (p[2] + p[3])) + ((p[4] + p[5]) + (p[6] + p[7]));
}

__device__ void row_stats(const float* __restrict__ row, int V, float inv_t, float* red, float& m, float& s) {
    // coalesced: thread t reads tokens t, t + blockDim, ... (a fixed order for the sum)
    float mx[8] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY, -INFINITY, -INFINITY, -INFINITY, -INFINITY};
    const int st = blockDim.x;
    int z = threadIdx.x;
    for (; z + 7 * st < V; z += 8 * st) {
#pragma unroll
        for (int k = 0; k < 8; ++k) mx[k] = fmaxf(mx[k], row[z + k * st]);
    }
#pragma unroll
    for (int k = 0; k < 8; ++k)
        if (z + k * st < V) mx[k] = fmaxf(mx[k], row[z + k * st]);
    m = block_max_f(fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])), fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))),
                    red);
    const float mm = m;
    s = block_sum_f(strided_sum([&](int zz) { return expf((row[zz] - mm) * inv_t); }, threadIdx.x, V, st), red);
}

// ---------------------------------------------------------------- law clusters

constexpr int LT = 512;             // threads of a law / verify CTA
constexpr int LW = LT / 32;         // its warps
constexpr int HB = 2048;            // radix bins per pass (11-bit digits)
constexpr int MAX_NC = 8;           // CTAs per cluster (portable limit)
constexpr float W_ONE = 2147483648.f;  // fixed-point scale of the top-p masses (2^31: one mass fits 32 bits)

// Per-CTA scratch in static shared memory.  Each `pub` slot is written once per
// launch by thread 0 and read by every CTA of the cluster after a cluster barrier.
enum { P_MAX, P_KCNT, P_KID, P_MK, P_PCNT, P_PID, P_TOT0, P_TOT1, N_PUB };
struct Scratch {
    unsigned long long pub[N_PUB];
    unsigned long long scan[LW];
    float fw[LW], fwex[LW];
    int sel_d, pick;
    unsigned long long sel_above;
};

// Rank key of a logit: larger logit -> larger key (-0 ranks as +0), and back.
__device__ __forceinline__ uint32_t rank_key(float x) { return f32_order_key(x == 0.f ? 0.f : x); }
__device__ __forceinline__ float key_value(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}
__device__ __forceinline__ bool is_kept(uint32_t key, int z, uint32_t tkey, int tid) {
    return key > tkey || (key == tkey && z <= tid);
}
// Filtered law weight exp((x - m) / T) of a kept token (by rank key), else 0.
__device__ __forceinline__ float law_weight(uint32_t key, int z, const LawStat& st, float inv_t) {
    return is_kept(key, z, st.tkey, st.tid) ? expf((key_value(key) - st.m) * inv_t) : 0.f;
}
// The same for a logit read from global memory.
__device__ __forceinline__ float law_weight_x(float x, int z, const LawStat& st, float inv_t) {
    return is_kept(rank_key(x), z, st.tkey, st.tid) ? expf((x - st.m) * inv_t) : 0.f;
}
__device__ __forceinline__ uint32_t fixed_mass(uint32_t key, float m, float inv_t) {
    return __float2uint_rn(expf((key_value(key) - m) * inv_t) * W_ONE);
}

__device__ __forceinline__ float clamp_u(float u) { return fminf(fmaxf(u, 0.f), 0.99999994f); }

template <typename T>
__device__ __forceinline__ T peer(cg::cluster_group& cl, T* p, int r) {
    return *cl.map_shared_rank(p, r);
}

// Exclusive prefix sum over the CTA's threads in thread order; *total = the sum.
__device__ unsigned long long block_excl_scan(unsigned long long v, Scratch& S, unsigned long long* total) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    unsigned long long inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long n = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += n;
    }
    __syncthreads();  // readers of the previous scan are done with S.scan
    if (lane == 31) S.scan[w] = inc;
    __syncthreads();
    const unsigned long long t = lane < LW ? S.scan[lane] : 0ull;
    unsigned long long ti = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long n = __shfl_up_sync(0xffffffffu, ti, o);
        if (lane >= o) ti += n;
    }
    *total = __shfl_sync(0xffffffffu, ti, LW - 1);
    return __shfl_sync(0xffffffffu, ti - t, w) + inc - v;
}

// Radix selection over the rank keys ks[0, n) of this CTA's chunk (tokens c0 + i),
// combined across the cluster.  W(z, key) is a token's weight (0: not a candidate),
// counted in bins of type BinT.  Finds the key t at which the candidates' weight,
// accumulated in rank order, first reaches `target`: weight(key > t) < target <=
// weight(key >= t); *above = weight(key > t).  Keys of candidates lie in [lo, hi].
// Digits of at most 11 bits from the top of (key - lo); `pass` alternates the two
// histogram buffers so that one cluster barrier per pass suffices.
template <typename BinT, class WF>
__device__ uint32_t radix_select(const uint32_t* ks, int n, int c0, uint32_t lo, uint32_t hi, double target,
                                 const WF& W, unsigned char* hist, int& pass, Scratch& S, cg::cluster_group& cl,
                                 int nc, double* above) {
    uint32_t base = lo;
    int L = hi > lo ? 32 - __clz(hi - lo) : 0;
    double acc = 0.0;
    while (L > 0) {
        const int bits = L < 11 ? L : 11, shift = L - bits;
        const unsigned long long span = 1ull << L;
        BinT* H = reinterpret_cast<BinT*>(hist + (pass & 1) * HB * sizeof(unsigned long long));
        ++pass;
        for (int i = threadIdx.x; i < HB; i += LT) H[i] = 0;
        if (threadIdx.x == 0) S.sel_d = -1;
        __syncthreads();
        for (int i = threadIdx.x; i < n; i += LT) {
            const uint32_t k = ks[i];
            if (k < base || (unsigned long long)(k - base) >= span) continue;
            const BinT w = (BinT)W(c0 + i, k);
            if (w) atomicAdd(&H[(k - base) >> shift], w);
        }
        cl.sync();
        // thread t sums bins 4t .. 4t+3 over the cluster's CTAs, in CTA order
        unsigned long long h0 = 0ull, h1 = 0ull, h2 = 0ull, h3 = 0ull;
#pragma unroll
        for (int r = 0; r < MAX_NC; ++r) {
            if (r < nc) {
                const BinT* P = cl.map_shared_rank(H, r) + 4 * threadIdx.x;
                if constexpr (sizeof(BinT) == 4) {
                    const uint4 a = *reinterpret_cast<const uint4*>(P);
                    h0 += a.x;
                    h1 += a.y;
                    h2 += a.z;
                    h3 += a.w;
                } else {
                    const ulonglong2 a = reinterpret_cast<const ulonglong2*>(P)[0];
                    const ulonglong2 b = reinterpret_cast<const ulonglong2*>(P)[1];
                    h0 += a.x;
                    h1 += a.y;
                    h2 += b.x;
                    h3 += b.y;
                }
            }
        }
        const unsigned long long mine = (h0 + h1) + (h2 + h3);
        unsigned long long total;
        const unsigned long long ex = block_excl_scan(mine, S, &total);
        const unsigned long long E = total - ex - mine;  // weight of the bins above this thread's
        if (mine && (double)E < target && target <= (double)(E + mine)) {
            // the crossing bin, from the highest of the four down
            unsigned long long a = E;
            int d = 4 * threadIdx.x;
            if (h3 && target <= (double)(a + h3)) {
                d += 3;
            } else {
                a += h3;
                if (h2 && target <= (double)(a + h2)) {
                    d += 2;
                } else {
                    a += h2;
                    if (h1 && target <= (double)(a + h1)) d += 1;
                    else a += h1;
                }
            }
            S.sel_d = d;
            S.sel_above = a;
        }
        __syncthreads();
        int d = S.sel_d;
        const unsigned long long ab = d >= 0 ? S.sel_above : 0ull;
        __syncthreads();
        if (d < 0) d = 0;  // target above the candidates' weight (not reached): keep them all
        target -= (double)ab;
        acc += (double)ab;
        base += (uint32_t)d << shift;
        L = shift;
    }
    *above = acc;
    return base;
}

// The id of the need-th (1-based, need >= 1) token in increasing id among the
// tokens of key t that pass `pred`, over the cluster's chunks (clamped to the
// last such token).  Uses the pub slots cnt_slot and id_slot.
template <class PF>
__device__ int tie_select(const uint32_t* ks, int n, int c0, uint32_t t, long long need, const PF& pred, int cnt_slot,
                          int id_slot, Scratch& S, cg::cluster_group& cl, int nc, int rank) {
    unsigned long long c = 0;
    for (int i = threadIdx.x; i < n; i += LT)
        if (ks[i] == t && pred(c0 + i)) ++c;
    unsigned long long tot;
    block_excl_scan(c, S, &tot);
    if (threadIdx.x == 0) {
        S.pub[cnt_slot] = tot;
        S.pub[id_slot] = (unsigned long long)-1;
    }
    cl.sync();
    long long ex = 0, ex_sel = 0, ex_last = 0;
    int rsel = -1, rlast = -1;
#pragma unroll
    for (int r = 0; r < MAX_NC; ++r) {
        if (r < nc) {
            const long long cr = (long long)peer(cl, &S.pub[cnt_slot], r);
            if (cr > 0) {
                rlast = r;
                ex_last = ex;
                if (rsel < 0 && ex + cr >= need) {
                    rsel = r;
                    ex_sel = ex;
                }
            }
            ex += cr;
        }
    }
    if (rsel < 0) {  // fewer ties than asked for: the last one
        rsel = rlast;
        ex_sel = ex_last;
        need = 1ll << 62;
    }
    if (rsel < 0) return -1;
    if (rank == rsel) {
        const long long local = need - ex_sel;
        const int R = (n + LT - 1) / LT;
        const int a0 = min(n, (int)threadIdx.x * R), a1 = min(n, a0 + R);
        unsigned long long ct = 0;
        for (int i = a0; i < a1; ++i)
            if (ks[i] == t && pred(c0 + i)) ++ct;
        unsigned long long ctot;
        const unsigned long long et = block_excl_scan(ct, S, &ctot);
        const long long want = local < (long long)ctot ? local : (long long)ctot;
        if (ct && (long long)et < want && want <= (long long)(et + ct)) {
            long long m = (long long)et;
            for (int i = a0; i < a1; ++i)
                if (ks[i] == t && pred(c0 + i) && ++m == want) {
                    S.pub[id_slot] = (unsigned long long)(c0 + i);
                    break;
                }
        }
    }
    cl.sync();
    return (int)(long long)peer(cl, &S.pub[id_slot], rsel);
}

// Weighted inverse-CDF draw over the row's tokens split across the cluster: CTA r
// owns its chunk (local indices i in [0, n), token c0 + i), warp k of each CTA a
// contiguous range of the chunk, lane l of the chosen warp a contiguous piece of
// that range.  Warp sums run lane-strided (coalesced) with a fixed combine, CTA
// and cluster totals fold in warp and CTA order.  Returns the row total (every
// CTA).  With `draw`, the CTA holding u * total sets S.pick to the drawn token
// (the last token of positive weight when rounding leaves u * total past every
// boundary) and every other CTA to -2; S.pick = -1 everywhere when the total is 0.
template <class WF>
__device__ float cluster_draw(const WF& w, int n, int c0, float u, bool draw, int slot, Scratch& S,
                              cg::cluster_group& cl, int nc, int rank) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int RW = ((n + LW - 1) / LW + 31) / 32 * 32;
    const int z0 = min(n, wid * RW), z1 = min(n, z0 + RW);
    __syncthreads();  // S.fw / S.pick of an earlier call are no longer read
    const float ws = warp_sum(strided_sum(w, z0 + lane, z1, 32));
    if (lane == 0) S.fw[wid] = ws;
    __syncthreads();
    if (threadIdx.x == 0) {
        float a = 0.f;
        for (int k = 0; k < LW; ++k) {
            S.fwex[k] = a;
            a += S.fw[k];
        }
        S.pub[slot] = __float_as_uint(a);
        S.pick = -2;
    }
    cl.sync();
    float total = 0.f;
#pragma unroll
    for (int r = 0; r < MAX_NC; ++r)
        if (r < nc) total += __uint_as_float((uint32_t)peer(cl, &S.pub[slot], r));
    if (!draw) return total;
    if (!(total > 0.f)) {
        if (threadIdx.x == 0) S.pick = -1;
        __syncthreads();
        return total;
    }
    const float target = u * total;
    int rsel = -1, rlast = -1;
    float ex_sel = 0.f, ex_last = 0.f;
    {
        float a = 0.f;
#pragma unroll
        for (int r = 0; r < MAX_NC; ++r) {
            const float tr = r < nc ? __uint_as_float((uint32_t)peer(cl, &S.pub[slot], r)) : 0.f;
            if (tr > 0.f) {
                rlast = r;
                ex_last = a;
                if (rsel < 0 && a + tr > target) {
                    rsel = r;
                    ex_sel = a;
                }
            }
            a += tr;
        }
    }
    if (rsel < 0) {
        rsel = rlast;
        ex_sel = ex_last;
    }
    if (rank != rsel) return total;
    const float tau = target - ex_sel;
    int ksel = -1, klast = -1;
    for (int k = 0; k < LW; ++k)
        if (S.fw[k] > 0.f) {
            klast = k;
            if (ksel < 0 && S.fwex[k] + S.fw[k] > tau) ksel = k;
        }
    if (ksel < 0) ksel = klast;
    if (wid == ksel) {
        const float tw = tau - S.fwex[ksel];
        const int R2 = (z1 - z0 + 31) / 32;
        const int a0 = min(z1, z0 + lane * R2), a1 = min(z1, a0 + R2);
        const float cs = strided_sum(w, a0, a1, 1);
        float inc = cs;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float v = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += v;
        }
        const float ex = inc - cs;
        const unsigned hit = __ballot_sync(0xffffffffu, cs > 0.f && ex + cs > tw);
        const unsigned pos = __ballot_sync(0xffffffffu, cs > 0.f);
        const int lsel = hit ? __ffs(hit) - 1 : 31 - __clz(pos);
        if (lane == lsel) {
            const float tl = tw - ex;
            float acc = 0.f;
            int found = -1, last = -1;
            for (int i = a0; i < a1; ++i) {
                const float wi = w(i);
                if (wi > 0.f) {
                    last = i;
                    acc += wi;
                    if (acc > tl) {
                        found = i;
                        break;
                    }
                }
            }
            S.pick = c0 + (found >= 0 ? found : last);
        }
    }
    __syncthreads();
    return total;
}

// The chunk of a law row owned by this CTA: tokens [c0, c0 + n).
__device__ __forceinline__ void chunk_of(int V, int nc, int rank, int& c0, int& n) {
    const int C = ((V + nc - 1) / nc + 3) / 4 * 4;
    c0 = min(V, rank * C);
    n = min(V, c0 + C) - c0;
}

// One law row: stage the chunk's rank keys, the row max, the top-k / top-p threshold
// and the kept sum; with `draw`, the inverse-CDF draw of the filtered law.
__device__ void law_row(const float* __restrict__ l, int V, float inv_t, int top_k, float top_p, float u, bool draw,
                        LawStat* stat, int* out, unsigned char* dsm, Scratch& S) {
    cg::cluster_group cl = cg::this_cluster();
    const int nc = (int)cl.num_blocks(), rank = (int)cl.block_rank();
    int c0, n;
    chunk_of(V, nc, rank, c0, n);
    unsigned char* hist = dsm;
    uint32_t* ks = reinterpret_cast<uint32_t*>(dsm + 2 * HB * sizeof(unsigned long long));
    // stage the keys (float4 loads where the chunk start is 16-byte aligned, SU in flight
    // per thread), with the chunk's highest and lowest key
    constexpr int SU = 8;
    uint32_t khi = 0u, klo = 0xffffffffu;
    const float* src = l + c0;
    int done = 0;
    if ((reinterpret_cast<uintptr_t>(src) & 15) == 0) {
        const int n4 = n >> 2;
        const float4* s4 = reinterpret_cast<const float4*>(src);
        for (int b = threadIdx.x; b < n4; b += SU * LT) {
            float4 v[SU];
#pragma unroll
            for (int k = 0; k < SU; ++k)
                if (b + k * LT < n4) v[k] = __ldg(s4 + b + k * LT);
#pragma unroll
            for (int k = 0; k < SU; ++k)
                if (b + k * LT < n4) {
                    const uint4 kk = make_uint4(rank_key(v[k].x), rank_key(v[k].y), rank_key(v[k].z), rank_key(v[k].w));
                    reinterpret_cast<uint4*>(ks)[b + k * LT] = kk;
                    khi = max(khi, max(max(kk.x, kk.y), max(kk.z, kk.w)));
                    klo = min(klo, min(min(kk.x, kk.y), min(kk.z, kk.w)));
                }
        }
        done = 4 * n4;
    }
    for (int b = done + threadIdx.x; b < n; b += SU * LT) {
        float v[SU];
#pragma unroll
        for (int k = 0; k < SU; ++k)
            if (b + k * LT < n) v[k] = __ldg(src + b + k * LT);
#pragma unroll
        for (int k = 0; k < SU; ++k)
            if (b + k * LT < n) {
                const uint32_t kk = rank_key(v[k]);
                ks[b + k * LT] = kk;
                khi = max(khi, kk);
                klo = min(klo, kk);
            }
    }
    // the cluster's highest and lowest key
    {
        const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            khi = max(khi, __shfl_xor_sync(0xffffffffu, khi, o));
            klo = min(klo, __shfl_xor_sync(0xffffffffu, klo, o));
        }
        if (lane == 0) S.scan[w] = ((unsigned long long)klo << 32) | khi;
        __syncthreads();
        if (threadIdx.x == 0) {
            uint32_t h = 0u, lo = 0xffffffffu;
            for (int k = 0; k < LW; ++k) {
                h = max(h, (uint32_t)S.scan[k]);
                lo = min(lo, (uint32_t)(S.scan[k] >> 32));
            }
            S.pub[P_MAX] = ((unsigned long long)lo << 32) | h;
        }
    }
    cl.sync();
    uint32_t hi = 0u, lo = 0xffffffffu;
#pragma unroll
    for (int r = 0; r < MAX_NC; ++r)
        if (r < nc) {
            const unsigned long long v = peer(cl, &S.pub[P_MAX], r);
            hi = max(hi, (uint32_t)v);
            lo = min(lo, (uint32_t)(v >> 32));
        }
    const float m = key_value(hi);
    LawStat st{m, 0.f, 0u, 0x7fffffff};  // keep every token
    int pass = 0;
    if (top_k > 0 && top_k < V) {
        double above;
        const uint32_t t = radix_select<uint32_t>(
            ks, n, c0, lo, hi, (double)top_k, [](int, uint32_t) { return 1u; }, hist, pass, S, cl, nc, &above);
        const long long need = (long long)top_k - (long long)above;
        st.tkey = t;
        st.tid = tie_select(ks, n, c0, t, need < 1 ? 1 : need, [](int) { return true; }, P_KCNT, P_KID, S, cl, nc, rank);
    }
    if (top_p < 1.f) {
        const LawStat sk = st;
        // the top-k set's fixed-point mass, then the key where p of it is reached
        unsigned long long mk = 0ull;
        for (int i = threadIdx.x; i < n; i += LT)
            if (is_kept(ks[i], c0 + i, sk.tkey, sk.tid)) mk += fixed_mass(ks[i], m, inv_t);
        unsigned long long mk_cta;
        block_excl_scan(mk, S, &mk_cta);
        if (threadIdx.x == 0) S.pub[P_MK] = mk_cta;
        cl.sync();
        unsigned long long Mk = 0ull;
#pragma unroll
        for (int r = 0; r < MAX_NC; ++r)
            if (r < nc) Mk += peer(cl, &S.pub[P_MK], r);
        const double target = (double)top_p * (double)Mk;
        double above;
        const uint32_t t = radix_select<unsigned long long>(
            ks, n, c0, sk.tkey > lo ? sk.tkey : lo, hi, target,
            [=](int z, uint32_t k) { return is_kept(k, z, sk.tkey, sk.tid) ? fixed_mass(k, m, inv_t) : 0u; }, hist,
            pass, S, cl, nc, &above);
        // equal keys have equal masses: the number of them to keep, in increasing id
        const unsigned long long wt = fixed_mass(t, m, inv_t);
        long long need = 1;
        if (wt > 0ull) {
            const double rest = target - above;
            need = (long long)ceil(rest / (double)wt);
            if (need < 1) need = 1;
            while (need > 1 && above + (double)((unsigned long long)(need - 1) * wt) >= target) --need;
            while (above + (double)((unsigned long long)need * wt) < target) ++need;
        }
        st.tkey = t;
        st.tid = tie_select(ks, n, c0, t, need, [=](int z) { return is_kept(t, z, sk.tkey, sk.tid); }, P_PCNT, P_PID, S,
                            cl, nc, rank);
    }
    const LawStat sf = st;
    const float total = cluster_draw([=](int i) { return law_weight(ks[i], c0 + i, sf, inv_t); }, n, c0, clamp_u(u),
                                     draw, P_TOT0, S, cl, nc, rank);
    if (rank == 0 && threadIdx.x == 0) {
        st.s = total;
        *stat = st;
    }
    if (draw && threadIdx.x == 0 && S.pick != -2) *out = S.pick;
    cl.sync();  // no CTA leaves while its shared memory may still be read
}

// Draft rows s*B + j, j = 1..B-1: the filtered law q_j and the proposal drawn from it.
// Grid (batch*(B-1), 1, nc), cluster (1, 1, nc).
__global__ void __launch_bounds__(LT, 2) draft_law_kernel(const float* __restrict__ dlogits, int V, int B,
                                                       const SampleParams* __restrict__ prm,
                                                       const float* __restrict__ u_draft, LawStat* __restrict__ dstat,
                                                       int* __restrict__ drafts) {
    extern __shared__ __align__(16) unsigned char dsm[];
    __shared__ Scratch S;
    pdl_wait();
    pdl_trigger();
    const int k = blockIdx.x, s = k / (B - 1), j = k % (B - 1) + 1;
    const int row = s * B + j;
    law_row(dlogits + (size_t)row * V, V, 1.f / prm->t_draft, prm->top_k, prm->top_p, u_draft[k], true, dstat + row,
            drafts + k, dsm, S);
}

// Target rows: the filtered laws p_j.  Grid (batch*B, 1, nc).
__global__ void __launch_bounds__(LT, 2) target_law_kernel(const float* __restrict__ logits, int V,
                                                        const SampleParams* __restrict__ prm,
                                                        LawStat* __restrict__ tstat) {
    extern __shared__ __align__(16) unsigned char dsm[];
    __shared__ Scratch S;
    pdl_wait();
    pdl_trigger();
    const int row = blockIdx.x;
    law_row(logits + (size_t)row * V, V, 1.f / prm->t_verify, prm->top_k, prm->top_p, 0.f, false, tstat + row, nullptr,
            dsm, S);
}

// One sequence per cluster: scan the proposals with eq. 6 under the filtered laws,
// emit a residual draw (eq. 7) at the first rejection or the bonus draw from
// p_{B-1}, then the round's bookkeeping (accepted count, emitted token = next
// anchor, length, context rows to append), written by the CTA that drew.
__global__ void __launch_bounds__(LT, 2) verify_sample_kernel(
    const float* __restrict__ logits, const float* __restrict__ dlogits, int V, int B,
    const SampleParams* __restrict__ prm, const int* __restrict__ proposal, const float* __restrict__ u_verify,
    const LawStat* __restrict__ tstat, const LawStat* __restrict__ dstat, int* __restrict__ n,
    int* __restrict__ anchor, int* __restrict__ accepted, int* __restrict__ bonus, int* __restrict__ ctx_row_seq,
    int* __restrict__ ctx_row_pos, uint32_t* err) {
    __shared__ Scratch S;
    __shared__ int a_s;
    pdl_wait();
    pdl_trigger();
    cg::cluster_group cl = cg::this_cluster();
    const int nc = (int)cl.num_blocks(), rank = (int)cl.block_rank();
    const int s = blockIdx.x;
    const float inv_td = 1.f / prm->t_draft, inv_tv = 1.f / prm->t_verify;
    const int* prop = proposal + (size_t)s * (B - 1);
    const float* u = u_verify + (size_t)s * B;
    if (threadIdx.x < 32) {
        // lane j decides proposal j (B - 1 <= 31); a = the number of leading accepts
        const int j = threadIdx.x;
        bool ok = false;
        if (j < B - 1) {
            const int y = prop[j];
            if (y < 0 || y >= V) {
                if (rank == 0) atomicOr(err, ERR_TOKEN_RANGE);
            } else {
                const LawStat ts = tstat[s * B + j], ds = dstat[s * B + j + 1];
                const float p = law_weight_x(logits[(size_t)(s * B + j) * V + y], y, ts, inv_tv) / ts.s;
                const float q = law_weight_x(dlogits[(size_t)(s * B + j + 1) * V + y], y, ds, inv_td) / ds.s;
                const float ratio = q > 0.f ? fminf(1.f, p / q) : 1.f;
                ok = clamp_u(u[j]) < ratio;
            }
        }
        const unsigned rej = __ballot_sync(0xffffffffu, !ok);  // lanes >= B-1 count as rejections
        if (j == 0) a_s = __ffs(rej) - 1;
    }
    __syncthreads();
    const int a = a_s;
    const float ue = clamp_u(u[B - 1]);
    int c0, cn;
    chunk_of(V, nc, rank, c0, cn);
    const float* lp = logits + (size_t)(s * B + a) * V + c0;
    const LawStat ts = tstat[s * B + a];
    auto p_of = [=](int i) { return law_weight_x(lp[i], c0 + i, ts, inv_tv) / ts.s; };
    float tot = 0.f;
    if (a < B - 1) {
        const float* lq = dlogits + (size_t)(s * B + a + 1) * V + c0;
        const LawStat ds = dstat[s * B + a + 1];
        tot = cluster_draw([=](int i) { return fmaxf(p_of(i) - law_weight_x(lq[i], c0 + i, ds, inv_td) / ds.s, 0.f); },
                           cn, c0, ue, true, P_TOT0, S, cl, nc, rank);
    }
    if (!(tot > 0.f)) cluster_draw(p_of, cn, c0, ue, true, P_TOT1, S, cl, nc, rank);  // bonus, or a residual of zero mass
    if (threadIdx.x == 0 && S.pick >= 0) {
        const int emit = S.pick, n0 = n[s];
        accepted[s] = a;
        bonus[s] = emit;
        anchor[s] = emit;
        n[s] = n0 + a + 1;
        for (int j = 0; j < B; ++j) {
            ctx_row_seq[s * B + j] = (j <= a) ? s : -1;
            ctx_row_pos[s * B + j] = n0 + j;
        }
    }
    cl.sync();
}

// Training loss rows: for sequence slots first .. first + n - 1 and block rows k = 1 .. B-1,
// out[i*(B-1) + k-1] = -log softmax(logits row)[label] = max + log sum exp(l - max) - l[label].
__global__ void __launch_bounds__(SNT) row_nll_kernel(const float* __restrict__ logits, int V, int B, int first,
                                                      const int* __restrict__ labels, float* __restrict__ out,
                                                      uint32_t* err) {
    pdl_wait();
    pdl_trigger();
    __shared__ float red[32];
    const int k = blockIdx.x, i = k / (B - 1), j = k % (B - 1) + 1;
    const float* l = logits + (size_t)((first + i) * B + j) * V;
    float m, sum;
    row_stats(l, V, 1.f, red, m, sum);
    if (threadIdx.x == 0) {
        const int y = labels[k];
        if (y < 0 || y >= V) {
            atomicOr(err, ERR_TOKEN_RANGE);
            out[k] = 0.f;
        } else {
            out[k] = m + logf(sum) - l[y];
        }
    }
}

}  // namespace

// CTAs per law row: one per 8192 tokens, at most a portable cluster of 8.
static int law_cluster_size(int V) {
    const int nc = (V + 8191) / 8192;
    return nc < 1 ? 1 : (nc > MAX_NC ? MAX_NC : nc);
}

// Dynamic shared memory of a law CTA: two radix histograms and the staged chunk of keys.
static size_t law_smem_bytes(int V) {
    const int nc = law_cluster_size(V);
    const size_t C = ((size_t)(V + nc - 1) / nc + 3) / 4 * 4;
    return 2 * HB * sizeof(unsigned long long) + C * sizeof(float);
}

bool sampling_vocab_ok(int V) { return V >= 1 && law_smem_bytes(V) + sizeof(Scratch) <= 227 * 1024; }

// Raises a law kernel's dynamic shared-memory limit to `bytes` (once per size increase).
static bool law_smem_attr(const void* fn, size_t bytes, size_t& set) {
    if (bytes <= set) return true;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) != cudaSuccess) return false;
    set = bytes;
    return true;
}

void draft_sample(const Launch& L, const float* dlogits, int V, int batch, int B, const SampleParams* prm,
                  const float* u_draft, LawStat* dstat, int* drafts) {
    if (batch <= 0 || B < 2) return;
    const int nc = law_cluster_size(V);
    const size_t sm = law_smem_bytes(V);
    static size_t set = 0;
    if (!law_smem_attr((const void*)draft_law_kernel, sm, set)) return L.fail();
    launch_k(L, draft_law_kernel, dim3(batch * (B - 1), 1, nc), dim3(LT), sm, nc, dlogits, V, B, prm, u_draft, dstat,
             drafts);
}

void verify_sample(const Launch& L, const float* logits, const float* dlogits, int V, int batch, int B,
                   const SampleParams* prm, const int* proposal, const float* u_verify, LawStat* tstat,
                   const LawStat* dstat, int* n, int* anchor, int* accepted, int* bonus, int* ctx_row_seq,
                   int* ctx_row_pos) {
    if (batch <= 0) return;
    const int nc = law_cluster_size(V);
    const size_t sm = law_smem_bytes(V);
    static size_t set = 0;
    if (!law_smem_attr((const void*)target_law_kernel, sm, set)) return L.fail();
    launch_k(L, target_law_kernel, dim3(batch * B, 1, nc), dim3(LT), sm, nc, logits, V, prm, tstat);
    launch_k(L, verify_sample_kernel, dim3(batch, 1, nc), dim3(LT), 0, nc, logits, dlogits, V, B, prm, proposal,
             u_verify, (const LawStat*)tstat, dstat, n, anchor, accepted, bonus, ctx_row_seq, ctx_row_pos, L.err);
}

void row_nll(const Launch& L, const float* logits, int V, int B, int first_seq, int n_seqs, const int* labels,
             float* out) {
    if (n_seqs <= 0 || B < 2) return;
    launch_k(L, row_nll_kernel, dim3(n_seqs * (B - 1)), dim3(SNT), 0, 1, logits, V, B, first_seq, labels, out, L.err);
}

}  // namespace dfl
