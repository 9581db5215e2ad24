// Temperature sampling of the draft-and-verify round (T > 0): speculative
// rejection sampling, "DFlash: Why a Diffusion Drafter Can Accelerate an
// Autoregressive Model" §4.2 (eq. 6-8) and Algorithm 1 (steps 2-3, 7-8, 10);
// "DFlash: Block Diffusion for Flash Speculative Decoding", Paper vs code
// "Sampling rule".
//
// Laws are softmax(logits / T) of fp32 logit rows: q from the draft head's
// rows 1..B-1, p from the verify head's rows 0..B-1 (p_j decides the proposal
// at block row j + 1).  Every draw is an inverse-CDF lookup of a caller-supplied
// uniform u in [0, 1): the lowest token z whose cumulative weight exceeds
// u * total.  One CTA handles one row (draws) or one sequence (acceptance and
// the emitted token); every pass over a row is coalesced and every sum is taken
// in one fixed order.
#include <math.h>

#include "launch.h"
#include "loss.h"

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
    for (int k = 0; z < end; z += stride, ++k) p[k & 7] += w(z);
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
    for (int k = 0; z < V; z += st, ++k) mx[k & 7] = fmaxf(mx[k & 7], row[z]);
    m = block_max_f(fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])), fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))),
                    red);
    const float mm = m;
    s = block_sum_f(strided_sum([&](int zz) { return expf((row[zz] - mm) * inv_t); }, threadIdx.x, V, st), red);
}

// Inverse-CDF draw over weights w(z) >= 0 (a functor), u in [0, 1): the lowest z whose
// cumulative weight exceeds u * total.  Warp k owns the contiguous token range
// [k R, (k + 1) R) and sums it coalesced; the warp sums are scanned in warp order; in
// the warp whose range holds u * total, lane l sums the contiguous sub-range
// [l R', (l + 1) R') of it, the lane sums are scanned in lane order, and the lane
// whose sub-range holds u * total walks it in token order.  Returns -1 when the
// total weight is 0.
template <class W>
__device__ int draw_inverse_cdf(const W& w, int V, float u, float* scan, int* pick) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const int R = ((V + nw - 1) / nw + 31) / 32 * 32;
    const int z0 = wid * R, z1 = min(V, z0 + R);
    const float ws = warp_sum(strided_sum(w, z0 + lane, z1, 32));
    if (lane == 0) scan[wid] = ws;
    if (threadIdx.x == 0) *pick = -1;
    __syncthreads();
    if (wid == 0) {
        const float wt = lane < nw ? scan[lane] : 0.f;
        float wi = wt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float n = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += n;
        }
        if (lane < nw) scan[32 + lane] = wi - wt;  // exclusive prefix of the warp sums
        if (lane == nw - 1) scan[64] = wi;         // total
    }
    __syncthreads();
    const float total = scan[64], excl = scan[32 + wid];
    const float target = u * total;
    if (total > 0.f && ws > 0.f && excl <= target && target < excl + ws) {
        const int R2 = (z1 - z0 + 31) / 32;
        const int c0 = min(z1, z0 + lane * R2), c1 = min(z1, c0 + R2);
        const float cs = strided_sum(w, c0, c1, 1);
        float inc = cs;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float n = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += n;
        }
        const float ex = excl + (inc - cs);
        const unsigned hit = __ballot_sync(0xffffffffu, cs > 0.f && ex <= target && target < ex + cs);
        int found = -1;
        if (hit && lane == __ffs(hit) - 1) {
            float acc = ex;
            int last = -1;
            for (int z = c0; z < c1; ++z) {
                const float wz = w(z);
                if (wz > 0.f) last = z;
                acc += wz;
                if (acc > target) {
                    found = z;
                    break;
                }
            }
            if (found < 0) found = last;
        }
        if (!hit) {
            // rounding put u * total past the lanes' boundaries: the last token with weight here
            for (int z = c1 - 1; z >= c0; --z)
                if (w(z) > 0.f) {
                    found = z;
                    break;
                }
        }
        if (found >= 0) atomicMax(pick, found);
    }
    __syncthreads();
    int r = *pick;
    if (r < 0 && total > 0.f) {
        // rounding left u * total past every warp boundary: the last token with weight
        int lastp = -1;
        for (int z = z1 - 1 - lane; z >= z0 && lastp < 0; z -= 32)
            if (w(z) > 0.f) lastp = z;
        atomicMax(pick, lastp);
        __syncthreads();
        r = *pick;
    }
    __syncthreads();
    return r;
}

__device__ __forceinline__ float clamp_u(float u) { return fminf(fmaxf(u, 0.f), 0.99999994f); }

// Draft rows s*B + j, j = 1..B-1: statistics of q_j and the proposal drawn from it.
__global__ void __launch_bounds__(SNT) draft_sample_kernel(const float* __restrict__ dlogits, int V, int B,
                                                           const float* __restrict__ temp,
                                                           const float* __restrict__ u_draft,
                                                           float2* __restrict__ dstat, int* __restrict__ drafts) {
    pdl_wait();
    pdl_trigger();
    __shared__ float red[72];
    __shared__ int pick;
    const int k = blockIdx.x, s = k / (B - 1), j = k % (B - 1) + 1;
    const int row = s * B + j;
    const float* l = dlogits + (size_t)row * V;
    const float inv_t = 1.f / temp[0];
    float m, sum;
    row_stats(l, V, inv_t, red, m, sum);
    if (threadIdx.x == 0) dstat[row] = make_float2(m, sum);
    const int z = draw_inverse_cdf([&](int zz) { return expf((l[zz] - m) * inv_t); }, V, clamp_u(u_draft[k]), red,
                                   &pick);
    if (threadIdx.x == 0) drafts[k] = z;
}

// Target rows: statistics of p_j.
__global__ void __launch_bounds__(SNT) target_stats_kernel(const float* __restrict__ logits, int V,
                                                           const float* __restrict__ temp,
                                                           float2* __restrict__ tstat) {
    pdl_wait();
    pdl_trigger();
    __shared__ float red[32];
    const int row = blockIdx.x;
    float m, sum;
    row_stats(logits + (size_t)row * V, V, 1.f / temp[1], red, m, sum);
    if (threadIdx.x == 0) tstat[row] = make_float2(m, sum);
}

// One sequence: scan the proposals with eq. 6, emit a residual draw (eq. 7) at the
// first rejection or the bonus draw from p_{B-1}, then the round's bookkeeping
// (accepted count, emitted token = next anchor, length, context rows to append).
__global__ void __launch_bounds__(SNT) verify_sample_kernel(
    const float* __restrict__ logits, const float* __restrict__ dlogits, int V, int B, const float* __restrict__ temp,
    const int* __restrict__ proposal, const float* __restrict__ u_verify, const float2* __restrict__ tstat,
    const float2* __restrict__ dstat, int* __restrict__ n, int* __restrict__ anchor, int* __restrict__ accepted,
    int* __restrict__ bonus, int* __restrict__ ctx_row_seq, int* __restrict__ ctx_row_pos, uint32_t* err) {
    pdl_wait();
    pdl_trigger();
    __shared__ float scan[72];
    __shared__ int pick, a_s;
    const int s = blockIdx.x;
    const float inv_td = 1.f / temp[0], inv_tv = 1.f / temp[1];
    const int* prop = proposal + (size_t)s * (B - 1);
    const float* u = u_verify + (size_t)s * B;
    if (threadIdx.x < 32) {
        // lane j decides proposal j (B - 1 <= 31); a = the number of leading accepts
        const int j = threadIdx.x;
        bool ok = false;
        if (j < B - 1) {
            const int y = prop[j];
            if (y < 0 || y >= V) {
                atomicOr(err, ERR_TOKEN_RANGE);
            } else {
                const float2 ts = tstat[s * B + j], ds = dstat[s * B + j + 1];
                const float p = expf((logits[(size_t)(s * B + j) * V + y] - ts.x) * inv_tv) / ts.y;
                const float q = expf((dlogits[(size_t)(s * B + j + 1) * V + y] - ds.x) * inv_td) / ds.y;
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
    const float* lp = logits + (size_t)(s * B + a) * V;
    const float2 ts = tstat[s * B + a];
    auto p_of = [&](int z) { return expf((lp[z] - ts.x) * inv_tv) / ts.y; };
    int emit = -1;
    if (a < B - 1) {
        const float* lq = dlogits + (size_t)(s * B + a + 1) * V;
        const float2 ds = dstat[s * B + a + 1];
        emit = draw_inverse_cdf(
            [&](int z) { return fmaxf(p_of(z) - expf((lq[z] - ds.x) * inv_td) / ds.y, 0.f); }, V, ue, scan, &pick);
    }
    if (emit < 0) emit = draw_inverse_cdf(p_of, V, ue, scan, &pick);  // bonus, or a residual of zero mass
    if (threadIdx.x == 0) {
        const int n0 = n[s];
        accepted[s] = a;
        bonus[s] = emit;
        anchor[s] = emit;
        n[s] = n0 + a + 1;
        for (int j = 0; j < B; ++j) {
            ctx_row_seq[s * B + j] = (j <= a) ? s : -1;
            ctx_row_pos[s * B + j] = n0 + j;
        }
    }
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

void draft_sample(const Launch& L, const float* dlogits, int V, int batch, int B, const float* temp,
                  const float* u_draft, float2* dstat, int* drafts) {
    if (batch <= 0 || B < 2) return;
    launch_k(L, draft_sample_kernel, dim3(batch * (B - 1)), dim3(SNT), 0, 1, dlogits, V, B, temp, u_draft, dstat,
             drafts);
}

void verify_sample(const Launch& L, const float* logits, const float* dlogits, int V, int batch, int B,
                   const float* temp, const int* proposal, const float* u_verify, float2* tstat, const float2* dstat,
                   int* n, int* anchor, int* accepted, int* bonus, int* ctx_row_seq, int* ctx_row_pos) {
    if (batch <= 0) return;
    launch_k(L, target_stats_kernel, dim3(batch * B), dim3(SNT), 0, 1, logits, V, temp, tstat);
    launch_k(L, verify_sample_kernel, dim3(batch), dim3(SNT), 0, 1, logits, dlogits, V, B, temp, proposal, u_verify,
             (const float2*)tstat, dstat, n, anchor, accepted, bonus, ctx_row_seq, ctx_row_pos, L.err);
}

void row_nll(const Launch& L, const float* logits, int V, int B, int first_seq, int n_seqs, const int* labels,
             float* out) {
    if (n_seqs <= 0 || B < 2) return;
    launch_k(L, row_nll_kernel, dim3(n_seqs * (B - 1)), dim3(SNT), 0, 1, logits, V, B, first_seq, labels, out, L.err);
}

}  // namespace dfl
