// Softmax attention over the paged KV cache for a group of query rows
// (CUDA-core kernel, used for fp32 storage; bf16 runs in attention_mma.cu).
//
// One CTA handles up to 64 query vectors = (rows of one sequence) x (the query
// heads sharing one KV head), over one contiguous range of keys (a split).
// Keys and values are staged tile by tile (64 keys) through shared memory and
// consumed with an online softmax in fp32.  Causal rows see keys [0, pos];
// non-causal rows (the draft block, "DFlash: Block Diffusion for Flash
// Speculative Decoding", Paper vs code "Attention pattern") see every key in
// [0, n_seq + extra).  When a group's keys are split over several CTAs, each
// writes (max, sum, unnormalised output) and a combine kernel merges the
// splits in split order, so the result does not depend on scheduling.
#include <math.h>

#include "launch.h"

namespace dfl {

namespace {

constexpr int QV = 64;   // query vectors per CTA
constexpr int KT = 64;   // keys per tile
constexpr int NT = 256;  // threads

struct AttnArgs {
    AttnParams p;
    int g;            // query heads per KV head
    int n_groups;
    int splits;
    int keys_per_split;
    float scale;
};

template <typename T, int HD>
__global__ void __launch_bounds__(NT) attn_kernel(AttnArgs a) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ float sm[];
    constexpr int QLD = HD + 1, SLD = KT + 1;   // padded rows: no shared-memory bank conflicts
    float* Qs = sm;                       // [QV][QLD]
    float* Ks = Qs + QV * QLD;            // [KT][HD + 1]
    float* Vs = Ks + KT * (HD + 1);       // [KT][HD]
    float* S = Vs + KT * HD;              // [QV][SLD]
    float* m_s = S + QV * SLD;            // [QV]
    float* l_s = m_s + QV;                // [QV]
    float* alpha = l_s + QV;              // [QV]
    __shared__ int lim_s[QV];

    const AttnParams& p = a.p;
    const int grp = blockIdx.x, kvh = blockIdx.y, split = blockIdx.z;
    const int g = a.g;
    const int r0 = grp * p.group_rows;
    const int nrows = min(p.group_rows, p.rows - r0);
    const int nv = nrows * g;
    const int tid = threadIdx.x;
    const int seq = p.row_seq[r0];

    // per query vector key limit (exclusive)
    int group_lim = 0;
    for (int v = tid; v < QV; v += NT) {
        int lim = 0;
        if (v < nv && seq >= 0) {
            const int r = r0 + v / g;
            if (p.row_seq[r] >= 0) lim = p.seq_len ? (p.seq_len[seq] + p.extra) : (p.row_pos[r] + 1);
        }
        lim_s[v] = lim;
        m_s[v] = -INFINITY;
        l_s[v] = 0.f;
    }
    __syncthreads();
    for (int v = 0; v < nv; ++v) group_lim = max(group_lim, lim_s[v]);
    const int k_begin = split * a.keys_per_split;
    const int k_end = min(k_begin + a.keys_per_split, group_lim);

    // queries, pre-scaled
    const T* q = reinterpret_cast<const T*>(p.q);
    for (int i = tid; i < QV * HD; i += NT) {
        const int v = i / HD, d = i % HD;
        float val = 0.f;
        if (v < nv) {
            const int r = r0 + v / g, h = kvh * g + v % g;
            val = to_f32(q[(size_t)r * p.H * HD + h * HD + d]) * a.scale;
        }
        Qs[v * QLD + d] = val;
    }

    // output accumulators: thread owns query vectors (2 vp, 2 vp + 1) and dims dg + 8 i
    const int vp = tid >> 3, dg = tid & 7;
    constexpr int DI = HD / 8;
    float acc0[DI], acc1[DI];
#pragma unroll
    for (int i = 0; i < DI; ++i) acc0[i] = acc1[i] = 0.f;

    const T* Kc = reinterpret_cast<const T*>(p.Kc);
    const T* Vc = reinterpret_cast<const T*>(p.Vc);
    __syncthreads();

    for (int kt = k_begin; kt < k_end; kt += KT) {
        // stage K and V tile
        for (int i = tid; i < KT * HD; i += NT) {
            const int kk = i / HD, d = i % HD;
            const int key = kt + kk;
            float kv = 0.f, vv = 0.f;
            if (key < k_end) {
                const long long off = kv_offset(p.kv, p.page_table, seq, key, kvh);
                kv = to_f32(Kc[off + d]);
                vv = to_f32(Vc[off + d]);
            }
            Ks[kk * (HD + 1) + d] = kv;
            Vs[kk * HD + d] = vv;
        }
        __syncthreads();
        // scores: thread -> query vector tid / 4, keys (tid % 4) + 4 j
        {
            const int v = tid >> 2, k0 = tid & 3;
            float s[KT / 4];
#pragma unroll
            for (int j = 0; j < KT / 4; ++j) s[j] = 0.f;
            const float* qrow = Qs + v * QLD;
            for (int d = 0; d < HD; ++d) {
                const float qd = qrow[d];
#pragma unroll
                for (int j = 0; j < KT / 4; ++j) s[j] += qd * Ks[(k0 + 4 * j) * (HD + 1) + d];
            }
            const int lim = lim_s[v];
#pragma unroll
            for (int j = 0; j < KT / 4; ++j) {
                const int key = kt + k0 + 4 * j;
                S[v * SLD + k0 + 4 * j] = (key < lim && key < k_end) ? s[j] : -INFINITY;
            }
        }
        __syncthreads();
        // online softmax: warp w handles query vectors w, w + 8, ...
        {
            const int lane = tid & 31, warp = tid >> 5;
            for (int v = warp; v < QV; v += NT / 32) {
                const float x0 = S[v * SLD + lane], x1 = S[v * SLD + lane + 32];
                const float mt = warp_max(fmaxf(x0, x1));
                const float mo = m_s[v];
                const float mn = fmaxf(mo, mt);
                float p0 = 0.f, p1 = 0.f, al = 1.f;
                if (mn != -INFINITY) {
                    p0 = (x0 == -INFINITY) ? 0.f : expf(x0 - mn);
                    p1 = (x1 == -INFINITY) ? 0.f : expf(x1 - mn);
                    al = (mo == -INFINITY) ? 0.f : expf(mo - mn);
                }
                const float ps = warp_sum(p0 + p1);
                S[v * SLD + lane] = p0;
                S[v * SLD + lane + 32] = p1;
                if (lane == 0) {
                    alpha[v] = al;
                    m_s[v] = mn;
                    l_s[v] = l_s[v] * al + ps;
                }
            }
        }
        __syncthreads();
        // O = O * alpha + P V
        {
            const int v0 = 2 * vp, v1 = 2 * vp + 1;
            const float a0 = alpha[v0], a1 = alpha[v1];
#pragma unroll
            for (int i = 0; i < DI; ++i) {
                acc0[i] *= a0;
                acc1[i] *= a1;
            }
            for (int kk = 0; kk < KT; ++kk) {
                const float p0 = S[v0 * SLD + kk], p1 = S[v1 * SLD + kk];
                const float* vr = Vs + kk * HD + dg;
#pragma unroll
                for (int i = 0; i < DI; ++i) {
                    const float vv = vr[8 * i];
                    acc0[i] += p0 * vv;
                    acc1[i] += p1 * vv;
                }
            }
        }
        __syncthreads();
    }

    // write
#pragma unroll
    for (int w = 0; w < 2; ++w) {
        const int v = 2 * vp + w;
        if (v >= nv) continue;
        const int r = r0 + v / g, h = kvh * g + v % g;
        if (p.row_seq[r] < 0) continue;
        float res[DI];
#pragma unroll
        for (int i = 0; i < DI; ++i) res[i] = w ? acc1[i] : acc0[i];
        if (a.splits == 1) {
            const float l = l_s[v];
            const float inv = l > 0.f ? 1.f / l : 0.f;
            T* o = reinterpret_cast<T*>(p.out) + (size_t)r * p.H * HD + h * HD;
#pragma unroll
            for (int i = 0; i < DI; ++i) o[dg + 8 * i] = from_f32<T>(res[i] * inv);
        } else {
            // workspace: O [splits][rows][H][HD], then (m, l) [splits][rows][H]
            const size_t base = ((size_t)split * p.rows + r) * p.H + h;
            float* O = p.ws + base * HD;
#pragma unroll
            for (int i = 0; i < DI; ++i) O[dg + 8 * i] = res[i];
            if (dg == 0) {
                float* ml = p.ws + (size_t)a.splits * p.rows * p.H * HD;
                ml[2 * base] = m_s[v];
                ml[2 * base + 1] = l_s[v];
            }
        }
    }
}

template <typename T, int HD>
__global__ void attn_combine_kernel(AttnArgs a) {
    pdl_wait();
    pdl_trigger();
    const AttnParams& p = a.p;
    const int r = blockIdx.x, h = blockIdx.y;
    if (p.row_seq[r] < 0) return;
    const float* ml = p.ws + (size_t)a.splits * p.rows * p.H * HD;
    float m = -INFINITY;
    for (int s = 0; s < a.splits; ++s) m = fmaxf(m, ml[2 * (((size_t)s * p.rows + r) * p.H + h)]);
    for (int d = threadIdx.x; d < HD; d += blockDim.x) {
        float num = 0.f, den = 0.f;
        for (int s = 0; s < a.splits; ++s) {
            const size_t base = ((size_t)s * p.rows + r) * p.H + h;
            const float ms = ml[2 * base], ls = ml[2 * base + 1];
            if (ms == -INFINITY) continue;
            const float w = expf(ms - m);
            num += w * p.ws[base * HD + d];
            den += w * ls;
        }
        T* o = reinterpret_cast<T*>(p.out) + (size_t)r * p.H * HD + h * HD;
        o[d] = from_f32<T>(den > 0.f ? num / den : 0.f);
    }
}

template <typename T, int HD>
void run(const Launch& L, const AttnParams& p) {
    AttnArgs a;
    a.p = p;
    a.g = p.H / p.Hkv;
    a.n_groups = (p.rows + p.group_rows - 1) / p.group_rows;
    a.scale = 1.f / sqrtf((float)HD);
    // split the keys so that small query counts still fill the GPU
    const int tiles = (p.max_keys + KT - 1) / KT;
    int splits = 1;
    const int ctas = a.n_groups * p.Hkv;
    if (ctas < 2 * 152 && tiles > 1) {
        splits = (2 * 152 + ctas - 1) / ctas;
        if (splits > tiles) splits = tiles;
        const size_t per = (size_t)p.rows * p.H * (HD + 2) * sizeof(float);
        const size_t cap = per ? p.ws_bytes / per : 0;
        if ((size_t)splits > cap) splits = (int)cap;
        if (splits < 1) splits = 1;
    }
    const int tiles_per_split = (tiles + splits - 1) / splits;
    a.keys_per_split = tiles_per_split * KT;
    a.splits = splits;
    if (p.group_rows * a.g > QV) return;  // the caller sizes groups to at most QV query vectors
    const size_t smem = (size_t)(QV * (HD + 1) + KT * (HD + 1) + KT * HD + QV * (KT + 1) + 3 * QV) * sizeof(float);
    static bool attr_set = false;
    if (!attr_set) {
        cudaFuncSetAttribute(attn_kernel<T, HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        attr_set = true;
    }
    dim3 grid(a.n_groups, p.Hkv, splits);
    launch_k(L, attn_kernel<T, HD>, grid, dim3(NT), smem, 1, a);
    if (splits > 1) launch_k(L, attn_combine_kernel<T, HD>, dim3(p.rows, p.H), dim3(HD), 0, 1, a);
}

}  // namespace

// fp32 storage: the CUDA-core kernel above.
template <>
void attention<float>(const Launch& L, const AttnParams& p) {
    if (p.rows <= 0) return;
    if (p.hd == 128)
        run<float, 128>(L, p);
    else
        run<float, 64>(L, p);
}

// bf16 storage: causal prefill chunks with 128-vector query groups run on tcgen05
// (attention_prefill.cu); the round's blocks (and anything else) on mma.sync
// (attention_mma.cu).
template <>
void attention<bf16>(const Launch& L, const AttnParams& p) {
    static int sms = 0;
    if (!sms) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (sms <= 0) sms = 148;
    }
    if (!p.seq_len && p.seq_div == 0 && p.hd == 128 && p.group_rows * (p.H / p.Hkv) == 128) {
        if (!attention_prefill_tc(L, p)) L.fail();
        return;
    }
    attention_mma(L, p, sms);
}

}  // namespace dfl
