// bf16 attention over the paged KV cache on the tensor cores (mma.sync
// m16n8k16), for query blocks of one sequence: the draft block (bidirectional
// over [context ; block], "DFlash: Block Diffusion for Flash Speculative
// Decoding", Paper vs code "Attention pattern") and the verify block (causal).
//
// A CTA owns up to 64 query vectors (the block rows of one sequence times the
// query heads sharing one KV head; four warps of 16) and one contiguous range
// of 64-key tiles.  A key tile is exactly one cache page, so it is one
// contiguous [64, head_dim] run in HBM; cp.async stages it (double-buffered)
// into XOR-swizzled shared memory read by ldmatrix.  Scores are fp32; the
// online softmax is fp32; P is split into bf16 hi + lo halves for the P.V
// product so the result keeps ~fp32 accuracy.
//
// The key tiles of a query group are dealt round-robin to S <= 16 CTAs that form
// a thread-block cluster (rank r takes tiles r, r + S, ...): the first page of
// every rank is known before the sequence length is read, so its K/V load
// starts one memory round trip earlier.  Each CTA parks (max, sum, unnormalised
// O) in shared memory and, after a cluster barrier, CTA r merges its share of
// the 64 query vectors over all ranks in rank order (deterministic), then writes
// the bf16 output.  The tiles a rank takes follow from the sequence's current
// length on the device, so the grid depends only on capacity.
#include <math.h>

#include "launch.h"

namespace dfl {

namespace {

constexpr int KT = 64;      // keys per tile (= cache page)
constexpr int NTHR = 128;   // 4 warps x 16 query vectors
constexpr int QV = 64;
constexpr int SMAX = 16;    // largest cluster (non-portable above 8)

__device__ __forceinline__ uint32_t s_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float* c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t crank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void csync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ float ld_peer(const float* local, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(s_u32(local)), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
}

__device__ __forceinline__ float4 ld_peer4(const float* local, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(s_u32(local)), "r"(rank));
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(remote)
                 : "memory");
    return v;
}

struct MmaArgs {
    AttnParams p;
    int g;        // query heads per KV head
    int splits;   // cluster size (<= SMAX)
    float scale_log2;  // log2(e) / sqrt(head_dim)
};

// Shared memory: K and V tiles, two stages each, rows of HD bf16 with the
// 16-byte chunks of row r XOR-swizzled by (r & 7).
template <int HD>
struct AttnSmem {
    static constexpr int TILE = KT * HD * 2;
    static constexpr int KV_BYTES = 4 * TILE;                  // K[2], V[2]
    static constexpr int PART = QV * HD * 4 + 2 * QV * 4;      // O, m, l (after the loop)
    static constexpr int TOTAL = (KV_BYTES > PART ? KV_BYTES : PART) + 128;
};

template <int HD>
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
    return (uint32_t)(row * (HD * 2) + ((chunk ^ (row & 7)) << 4));
}

template <int HD>
__global__ void __launch_bounds__(NTHR) attn_mma_kernel(MmaArgs a) {
    using SM = AttnSmem<HD>;
    constexpr int CH = HD / 8;         // 16-byte chunks per row
    constexpr int NB_O = HD / 8;       // n-blocks of the output
    extern __shared__ __align__(128) uint8_t sm[];
    __shared__ int lim_s[QV];
    __shared__ int glim_s;

    const AttnParams& p = a.p;
    const int grp = blockIdx.x, kvh = blockIdx.y;
    const int S = a.splits;
    const uint32_t rank = (S > 1) ? crank() : 0u;
    const int g = a.g;
    const int r0 = grp * p.group_rows;
    const int nrows = min(p.group_rows, p.rows - r0);
    const int nv = nrows * g;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // sequence of this group: from the row layout when it is sequence-major, else from row_seq
    // (read after the dependency wait)
    int seq = p.seq_div > 0 ? r0 / p.seq_div : -1;

    const uint8_t* Kc = reinterpret_cast<const uint8_t*>(p.Kc);
    const uint8_t* Vc = reinterpret_cast<const uint8_t*>(p.Vc);
    uint8_t* Ks = sm;
    uint8_t* Vs = sm + 2 * SM::TILE;

    auto load_tile = [&](int t, int stage) {
        // page of tile t holds keys [64 t, 64 t + 64) of this sequence
        const int page = p.page_table[seq * p.kv.pages_per_seq + t];
        const size_t off = ((size_t)page * p.kv.n_kv_heads + kvh) * (size_t)KT * HD * 2;
        const uint8_t* ksrc = Kc + off;
        const uint8_t* vsrc = Vc + off;
        uint8_t* kd = Ks + stage * SM::TILE;
        uint8_t* vd = Vs + stage * SM::TILE;
        for (int i = tid; i < KT * CH; i += NTHR) {
            const int r = i / CH, c = i % CH;
            cp_async16(kd + swz<HD>(r, c), ksrc + (size_t)i * 16);
            cp_async16(vd + swz<HD>(r, c), vsrc + (size_t)i * 16);
        }
        cp_commit();
    };
    // this rank's first tile (index `rank`): when it lies inside the sequence's stable keys
    // it loads before the dependency wait, under the tail of the kernel that writes Q and
    // the block's K/V; otherwise right after the wait, while the key limits are read (it is
    // dropped below if the sequence is shorter)
    // key limit of each query vector (causal: its position + 1; else seq_len + extra)
    auto key_limits = [&]() {
        if (tid == 0) glim_s = 0;
        __syncthreads();
        for (int v = tid; v < QV; v += NTHR) {
            int lim = 0;
            if (v < nv && seq >= 0) {
                const int r = r0 + v / g;
                if (p.row_seq[r] >= 0) lim = p.seq_len ? (p.seq_len[seq] + p.extra) : (p.row_pos[r] + 1);
            }
            lim_s[v] = lim;
            atomicMax(&glim_s, lim);
        }
        __syncthreads();
    };
    bool loaded = false;
    // round passes (stable_len set): the rows' metadata and lengths were written at the start of
    // the pass or earlier, so the limits are read before the dependency wait too
    const bool early = p.stable_len != nullptr && p.seq_div > 0;
    if (early) {
        if ((int)rank < p.kv.pages_per_seq && ((int)rank + 1) * KT <= p.stable_len[seq]) {
            load_tile((int)rank, 0);
            loaded = true;
        }
        key_limits();
    }
    pdl_wait();
    pdl_trigger();
    if (p.seq_div <= 0) seq = p.row_seq[r0];
    if (!loaded && seq >= 0 && (int)rank < p.kv.pages_per_seq) load_tile((int)rank, 0);
    if (!early) key_limits();
    const int glim = glim_s;
    const int tiles = (glim + KT - 1) / KT;

    // Q fragments (A operand), rows 16 warp + lane/4 (+8), head dims in k-steps of 16
    const int qa = 16 * warp + (lane >> 2), qb = qa + 8;
    uint32_t qf[HD / 16][4];
    {
        const __nv_bfloat16* q = reinterpret_cast<const __nv_bfloat16*>(p.q);
        auto qptr = [&](int v) -> const uint32_t* {
            const int r = r0 + v / g, h = kvh * g + v % g;
            return reinterpret_cast<const uint32_t*>(q + (size_t)r * p.H * HD + (size_t)h * HD);
        };
        const uint32_t* pa = qa < nv ? qptr(qa) : nullptr;
        const uint32_t* pb = qb < nv ? qptr(qb) : nullptr;
        const int c2 = lane & 3;  // column pair within 8
#pragma unroll
        for (int ks = 0; ks < HD / 16; ++ks) {
            qf[ks][0] = pa ? pa[ks * 8 + c2] : 0u;
            qf[ks][1] = pb ? pb[ks * 8 + c2] : 0u;
            qf[ks][2] = pa ? pa[ks * 8 + 4 + c2] : 0u;
            qf[ks][3] = pb ? pb[ks * 8 + 4 + c2] : 0u;
        }
    }
    const int lim_a = qa < nv ? lim_s[qa] : 0;
    const int lim_b = qb < nv ? lim_s[qb] : 0;

    float o[NB_O][4];
#pragma unroll
    for (int i = 0; i < NB_O; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;

    for (int it = 0;; ++it) {
        const int t = (int)rank + it * S;
        if (t >= tiles) break;
        const int stage = it & 1;
        if (t + S < tiles) {
            load_tile(t + S, stage ^ 1);
            cp_wait<1>();
        } else {
            cp_wait<0>();
        }
        __syncthreads();
        const uint32_t kbase = s_u32(Ks + stage * SM::TILE);
        const uint32_t vbase = s_u32(Vs + stage * SM::TILE);

        // S = Q K^T for 64 keys: n-block nb covers keys 8 nb .. 8 nb + 7
        float sc[8][4];
#pragma unroll
        for (int nb = 0; nb < 8; ++nb) {
            sc[nb][0] = sc[nb][1] = sc[nb][2] = sc[nb][3] = 0.f;
            const int krow = 8 * nb + (lane & 7);
#pragma unroll
            for (int kp = 0; kp < HD / 32; ++kp) {
                // four 8x8 matrices: head-dim chunks 4 kp .. 4 kp + 3 of keys krow
                uint32_t b0, b1, b2, b3;
                ldsm_x4(kbase + swz<HD>(krow, 4 * kp + (lane >> 3)), b0, b1, b2, b3);
                mma_bf16(sc[nb], qf[2 * kp][0], qf[2 * kp][1], qf[2 * kp][2], qf[2 * kp][3], b0, b1);
                mma_bf16(sc[nb], qf[2 * kp + 1][0], qf[2 * kp + 1][1], qf[2 * kp + 1][2], qf[2 * kp + 1][3], b2, b3);
            }
        }
        // scale, mask, online softmax (base 2)
        const int kbase_idx = t * KT + 2 * (lane & 3);
        float mx_a = -INFINITY, mx_b = -INFINITY;
#pragma unroll
        for (int nb = 0; nb < 8; ++nb) {
            const int k0 = kbase_idx + 8 * nb;
            sc[nb][0] = (k0 < lim_a) ? sc[nb][0] * a.scale_log2 : -INFINITY;
            sc[nb][1] = (k0 + 1 < lim_a) ? sc[nb][1] * a.scale_log2 : -INFINITY;
            sc[nb][2] = (k0 < lim_b) ? sc[nb][2] * a.scale_log2 : -INFINITY;
            sc[nb][3] = (k0 + 1 < lim_b) ? sc[nb][3] * a.scale_log2 : -INFINITY;
            mx_a = fmaxf(mx_a, fmaxf(sc[nb][0], sc[nb][1]));
            mx_b = fmaxf(mx_b, fmaxf(sc[nb][2], sc[nb][3]));
        }
        mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 1));
        mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 2));
        mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 1));
        mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 2));
        const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
        const float al_a = (mn_a == -INFINITY) ? 1.f : exp2f(m_a - mn_a);
        const float al_b = (mn_b == -INFINITY) ? 1.f : exp2f(m_b - mn_b);
        float sum_a = 0.f, sum_b = 0.f;
#pragma unroll
        for (int nb = 0; nb < 8; ++nb) {
            sc[nb][0] = (sc[nb][0] == -INFINITY) ? 0.f : exp2f(sc[nb][0] - mn_a);
            sc[nb][1] = (sc[nb][1] == -INFINITY) ? 0.f : exp2f(sc[nb][1] - mn_a);
            sc[nb][2] = (sc[nb][2] == -INFINITY) ? 0.f : exp2f(sc[nb][2] - mn_b);
            sc[nb][3] = (sc[nb][3] == -INFINITY) ? 0.f : exp2f(sc[nb][3] - mn_b);
            sum_a += sc[nb][0] + sc[nb][1];
            sum_b += sc[nb][2] + sc[nb][3];
        }
        sum_a += __shfl_xor_sync(0xffffffffu, sum_a, 1);
        sum_a += __shfl_xor_sync(0xffffffffu, sum_a, 2);
        sum_b += __shfl_xor_sync(0xffffffffu, sum_b, 1);
        sum_b += __shfl_xor_sync(0xffffffffu, sum_b, 2);
        l_a = l_a * al_a + sum_a;
        l_b = l_b * al_b + sum_b;
        m_a = mn_a;
        m_b = mn_b;
#pragma unroll
        for (int i = 0; i < NB_O; ++i) {
            o[i][0] *= al_a;
            o[i][1] *= al_a;
            o[i][2] *= al_b;
            o[i][3] *= al_b;
        }
        // O += P V with P split into bf16 hi + lo halves (P ~ hi + lo to ~16 bits);
        // keys 16 kk .. 16 kk + 15 per k-step
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const float* s0 = sc[2 * kk];
            const float* s1 = sc[2 * kk + 1];
            const float src[8] = {s0[0], s0[1], s0[2], s0[3], s1[0], s1[1], s1[2], s1[3]};
            // A fragment order: (rows a, keys lo) (rows b, keys lo) (rows a, keys hi) (rows b, keys hi)
            uint32_t ph[4], pl[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                ph[e] = pack_bf16(src[2 * e], src[2 * e + 1]);
                const float hx = __uint_as_float(ph[e] << 16), hy = __uint_as_float(ph[e] & 0xFFFF0000u);
                pl[e] = pack_bf16(src[2 * e] - hx, src[2 * e + 1] - hy);
            }
            const int vrow = 16 * kk + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
            for (int hb = 0; hb < NB_O; hb += 2) {
                // matrices: (keys 0-7, dims hb), (keys 8-15, dims hb), (keys 0-7, dims hb+1), (keys 8-15, dims hb+1)
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(vbase + swz<HD>(vrow, hb + (lane >> 4)), b0, b1, b2, b3);
                mma_bf16(o[hb], ph[0], ph[1], ph[2], ph[3], b0, b1);
                mma_bf16(o[hb], pl[0], pl[1], pl[2], pl[3], b0, b1);
                mma_bf16(o[hb + 1], ph[0], ph[1], ph[2], ph[3], b2, b3);
                mma_bf16(o[hb + 1], pl[0], pl[1], pl[2], pl[3], b2, b3);
            }
        }
        __syncthreads();  // the stage is overwritten by the next prefetch
    }
    cp_wait<0>();  // an early tile load that was not needed must land before the memory is reused
    __syncthreads();

    // ---- merge the splits and write
    float* Op = reinterpret_cast<float*>(sm);       // [QV][HD]
    float* Mp = Op + QV * HD;                       // [QV]
    float* Lp = Mp + QV;                            // [QV]
    if (S > 1) {
        // this thread's accumulators: rows qa / qb, dims 8 i + 2 (lane & 3) + {0, 1}
#pragma unroll
        for (int i = 0; i < NB_O; ++i) {
            const int d = 8 * i + 2 * (lane & 3);
            *reinterpret_cast<float2*>(Op + qa * HD + d) = make_float2(o[i][0], o[i][1]);
            *reinterpret_cast<float2*>(Op + qb * HD + d) = make_float2(o[i][2], o[i][3]);
        }
        if ((lane & 3) == 0) {
            Mp[qa] = m_a;
            Lp[qa] = l_a;
            Mp[qb] = m_b;
            Lp[qb] = l_b;
        }
        csync();
        // rank r merges query vectors [r * vper, (r + 1) * vper): each thread takes one
        // (vector, 4-dim chunk), loads every rank's (max, sum, O chunk) at once (one DSMEM
        // round trip) and combines them in rank order
        const int vper = QV / S + ((QV % S) ? 1 : 0);
        const int v0 = (int)rank * vper, v1 = min(QV, v0 + vper);
        __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out);
        constexpr int C4 = HD / 4;
        for (int idx = tid; idx < (v1 - v0) * C4; idx += NTHR) {
            const int v = v0 + idx / C4, d = 4 * (idx % C4);
            const int r = r0 + v / g, h = kvh * g + v % g;
            const bool live = v < nv && p.row_seq[r] >= 0;
            float ms[SMAX], ls[SMAX];
            float4 x[SMAX];
#pragma unroll
            for (int q = 0; q < SMAX; ++q) {
                const bool in = q < S;
                ms[q] = in ? ld_peer(Mp + v, (uint32_t)q) : -INFINITY;
                ls[q] = in ? ld_peer(Lp + v, (uint32_t)q) : 0.f;
                x[q] = in ? ld_peer4(Op + v * HD + d, (uint32_t)q) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            float mstar = -INFINITY;
#pragma unroll
            for (int q = 0; q < SMAX; ++q) mstar = fmaxf(mstar, ms[q]);
            float den = 0.f;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int q = 0; q < SMAX; ++q) {
                const float e = ms[q] != -INFINITY ? exp2f(ms[q] - mstar) : 0.f;
                den += e * ls[q];
                acc.x += e * x[q].x;
                acc.y += e * x[q].y;
                acc.z += e * x[q].z;
                acc.w += e * x[q].w;
            }
            const float inv = den > 0.f ? 1.f / den : 0.f;
            if (live) {
                __nv_bfloat16* dst = out + (size_t)r * p.H * HD + (size_t)h * HD + d;
                *reinterpret_cast<__nv_bfloat162*>(dst) = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
                *reinterpret_cast<__nv_bfloat162*>(dst + 2) = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
            }
        }
        csync();
    } else {
        __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out);
        const float ia = l_a > 0.f ? 1.f / l_a : 0.f, ib = l_b > 0.f ? 1.f / l_b : 0.f;
        const bool wa = qa < nv && p.row_seq[r0 + qa / g] >= 0;
        const bool wb = qb < nv && p.row_seq[r0 + qb / g] >= 0;
        __nv_bfloat16* oa = wa ? out + (size_t)(r0 + qa / g) * p.H * HD + (size_t)(kvh * g + qa % g) * HD : nullptr;
        __nv_bfloat16* ob = wb ? out + (size_t)(r0 + qb / g) * p.H * HD + (size_t)(kvh * g + qb % g) * HD : nullptr;
#pragma unroll
        for (int i = 0; i < NB_O; ++i) {
            const int d = 8 * i + 2 * (lane & 3);
            if (oa) *reinterpret_cast<__nv_bfloat162*>(oa + d) = __floats2bfloat162_rn(o[i][0] * ia, o[i][1] * ia);
            if (ob) *reinterpret_cast<__nv_bfloat162*>(ob + d) = __floats2bfloat162_rn(o[i][2] * ib, o[i][3] * ib);
        }
    }
}

template <int HD>
void run_mma(const Launch& L, const AttnParams& p, int sms) {
    MmaArgs a;
    a.p = p;
    a.g = p.H / p.Hkv;
    const int n_groups = (p.rows + p.group_rows - 1) / p.group_rows;
    a.scale_log2 = 1.4426950408889634f / sqrtf((float)HD);
    // cluster size from the capacity (so the launch is the same every round)
    const int cap_tiles = (p.max_keys + KT - 1) / KT;
    const int base = n_groups * p.Hkv;
    int S = 1;
    // (each rank keeps at least two tiles of capacity: below that the wider merge costs
    // more than the tile it saves)
    while (S < SMAX && S * 2 <= cap_tiles && base * S * 2 <= 2 * sms) S *= 2;
    a.splits = S;
    using SM = AttnSmem<HD>;
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(attn_mma_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, SM::TOTAL);
        cudaFuncSetAttribute(attn_mma_kernel<HD>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        attr = true;
    }
    launch_k(L, attn_mma_kernel<HD>, dim3(n_groups, p.Hkv, S), dim3(NTHR), (size_t)SM::TOTAL, S, a);
}

}  // namespace

// bf16 attention on mma.sync; the query group must hold at most 64 query vectors
// (group_rows * H / H_kv <= 64) and the cache page must be 64 tokens.
void attention_mma(const Launch& L, const AttnParams& p, int sms) {
    if (p.rows <= 0) return;
    if (p.hd == 128) run_mma<128>(L, p, sms);
    else run_mma<64>(L, p, sms);
}

}  // namespace dfl
