// Causal attention of a prefill chunk on the 5th-generation tensor cores
// (tcgen05 + TMEM), head_dim 128, bf16 cache.  The target prefill of
// "DFlash: Block Diffusion for Flash Speculative Decoding" (Method, Inference
// step 1) is a plain causal forward over the prompt; this kernel is its
// attention for chunks of many query rows, where the work is a dense
// contraction (the round's blocks of 16 rows use attention_mma.cu).
//
// A CTA owns 128 query vectors: 128 / g positions of one sequence times the g
// query heads of one KV head.  Query vector v is TMEM lane v; NSPLIT threads
// share it, v, v + 128, ... (warps q, q + 4, ... use the same TMEM lane
// quadrant): part i takes key columns [i 64 / NSPLIT, (i + 1) 64 / NSPLIT) of each
// tile and O columns [i 128 / NSPLIT, (i + 1) 128 / NSPLIT), and the parts
// exchange their tile maxima through shared memory (a named barrier per lane
// quadrant).  The CTA walks the
// 64-key tiles (= cache pages) 0 .. ceil(max position / 64) in order, with a
// software pipeline per tile t:
//   - S_{t+1} = Q K_{t+1}^T is issued on the tensor cores before the softmax of
//     tile t runs (S is double-buffered in TMEM: 2 x 64 columns);
//   - the softmax of tile t is online (fp32, base 2) with a lazy reference max
//     that only moves when a new score exceeds it by more than 2^8, so the
//     running O (128 TMEM columns) is rescaled rarely;
//   - P_t goes to shared memory as bf16 hi + lo halves (P ~ hi + lo to ~16 bits,
//     so the product keeps near-fp32 accuracy) and O += P_hi V_t + P_lo V_t is
//     issued (V as the MN-major B operand);
//   - K/V of tile t + 3 load (cp.async) into the ring stage that tile t - 1 has
//     released (four stages).
// One thread issues every tcgen05.mma; completion is tracked by mbarriers.  Every
// wait is bounded: one that runs out records ERR_TIMEOUT, the thread skips its
// later waits (every thread still meets every barrier), the output is not
// written, and the CTA releases its TMEM and returns.
#include <math.h>

#include "launch.h"
#include "tcgen05.cuh"

namespace dfl {

namespace {

using namespace tc;

constexpr int KT = 64;       // keys per tile = cache page
constexpr int HD = 128;      // head dim
constexpr int QM = 128;      // query vectors per CTA (MMA M)
constexpr int NSPLIT = 4;    // threads per query vector (warps q, q + 4, ... share a TMEM lane quadrant)
constexpr int NT = 128 * NSPLIT;
constexpr int KH = KT / NSPLIT;   // key columns per thread of a tile
constexpr int OH = 128 / NSPLIT;  // O columns per thread
constexpr int RING = 4;      // K/V ring stages

constexpr int Q_REG = QM * 128;       // 16 KB: one 64-dim half of the 128 query rows
constexpr int KV_REG = KT * 128;      // 8 KB: one 64-dim half of a 64-key tile
constexpr int Q_OFF = 0;                              // Q: 2 regions
constexpr int K_OFF = Q_OFF + 2 * Q_REG;              // K ring: RING x 2 regions
constexpr int V_OFF = K_OFF + RING * 2 * KV_REG;      // V ring
constexpr int P_OFF = V_OFF + RING * 2 * KV_REG;      // P hi, P lo: [128 rows][64 keys] bf16 each
constexpr int BAR_OFF = P_OFF + 2 * QM * 128;
constexpr int SMEM = BAR_OFF + 64 + 1024;             // + alignment slack

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// byte offset of 16-byte chunk c (0..7) of row r in a 128-byte-swizzled region
__device__ __forceinline__ uint32_t swz(int r, int c) { return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)); }

struct PfArgs {
    AttnParams p;
    int g;
    float scale_log2;  // log2(e) / sqrt(head_dim)
    uint32_t* err;
};

__global__ void __launch_bounds__(NT, 1) attn_prefill_tc_kernel(PfArgs a) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* sm = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const uint32_t sb = smem_u32(sm);
    uint64_t* bar_s = reinterpret_cast<uint64_t*>(sm + BAR_OFF);  // [2]: S buffer 0 / 1 complete
    uint64_t* bar_o = bar_s + 2;                                  // P.V complete
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_s + 3);
    __shared__ int glim_s;
    __shared__ float xch_s[NSPLIT][QM];  // the parts of each query vector: tile max, final sum

    const AttnParams& p = a.p;
    const int grp = gridDim.x - 1 - blockIdx.x;  // later positions (more key tiles) first
    const int kvh = blockIdx.y;
    const int g = a.g;
    const int r0 = grp * p.group_rows;
    const int nrows = min(p.group_rows, p.rows - r0);
    const int nv = nrows * g;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int v = tid & (QM - 1), half = tid >> 7;  // query vector (TMEM lane) and its key / O part
    const int seq = p.seq_div > 0 ? r0 / p.seq_div : p.row_seq[r0];

    if (warp == 0) {
        tmem_alloc(tmem_slot, 256);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&bar_s[0], 1);
        mbar_init(&bar_s[1], 1);
        mbar_init(bar_o, 1);
        mbar_fence_init();
        glim_s = 0;
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t t_lane = (uint32_t)(32 * (warp & 3)) << 16;
    const uint32_t tO = tmem + t_lane + 128 + OH * half;  // this thread's O columns (of 128 .. 255)

    // causal key limit of this thread's query vector
    int lim = 0;
    if (v < nv && seq >= 0) {
        const int r = r0 + v / g;
        if (p.row_seq[r] >= 0) lim = p.row_pos[r] + 1;
    }
    atomicMax(&glim_s, lim);
    // Q into the swizzled A operand (padding rows zero): each part copies 16 / NSPLIT of the
    // row's sixteen 16-byte chunks
    {
        constexpr int QC = 16 / NSPLIT;
        const uint4* src = nullptr;
        if (v < nv) {
            const int r = r0 + v / g, h = kvh * g + v % g;
            src = reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(p.q) + (size_t)r * p.H * HD +
                                                 (size_t)h * HD);
        }
#pragma unroll
        for (int i = 0; i < QC; ++i) {
            const int ch = QC * half + i;
            const uint4 x = src ? src[ch] : make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4*>(sm + Q_OFF + (ch >> 3) * Q_REG + swz(v, ch & 7)) = x;
        }
    }
    __syncthreads();
    const int n = seq >= 0 ? (glim_s + KT - 1) / KT : 0;

    const uint8_t* Kc = reinterpret_cast<const uint8_t*>(p.Kc);
    const uint8_t* Vc = reinterpret_cast<const uint8_t*>(p.Vc);
    // K/V of tile t into ring stage t % RING; always one commit group (possibly empty)
    auto load_tile = [&](int t) {
        if (t < n) {
            const int stage = t % RING;
            const int page = p.page_table[seq * p.kv.pages_per_seq + t];
            const size_t off = ((size_t)page * p.kv.n_kv_heads + kvh) * (size_t)KT * HD * 2;
            const uint8_t* ks = Kc + off;
            const uint8_t* vs = Vc + off;
            const uint32_t kd = sb + K_OFF + stage * 2 * KV_REG, vd = sb + V_OFF + stage * 2 * KV_REG;
            for (int i = tid; i < KT * 16; i += NT) {
                const int r = i >> 4, ch = i & 15;
                const uint32_t o = (uint32_t)((ch >> 3) * KV_REG) + swz(r, ch & 7);
                cp_async16(kd + o, ks + (size_t)i * 16);
                cp_async16(vd + o, vs + (size_t)i * 16);
            }
        }
        cp_commit();
    };
    constexpr uint32_t ID_S = idesc_bf16(QM, KT), ID_O = idesc_bf16(QM, HD, true);
    auto issue_s = [&](int t) {  // S_t = Q K_t^T into S buffer t & 1 (thread 0)
        const uint32_t qa = sb + Q_OFF, kb = sb + K_OFF + (t % RING) * 2 * KV_REG;
        const uint32_t d = tmem + (uint32_t)((t & 1) * KT);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)
            umma_bf16(d, sw128_desc(qa + (kk >> 2) * Q_REG + (kk & 3) * 32),
                      sw128_desc(kb + (kk >> 2) * KV_REG + (kk & 3) * 32), ID_S, kk > 0 ? 1u : 0u);
        umma_commit(&bar_s[t & 1]);
    };

    load_tile(0);
    load_tile(1);
    load_tile(2);
    float m_run = -INFINITY, l_run = 0.f;
    bool okw = true;  // a wait that ran out: later waits are skipped, barriers are still met
    auto wait = [&](uint64_t* bar, uint32_t parity) {
        if (okw && !mbar_wait(bar, parity, a.err)) okw = false;
    };
    if (n > 0) {
        cp_wait<2>();  // tile 0 landed
        fence_proxy_async();
        fence_before();
        __syncthreads();
        if (tid == 0) {
            fence_after();
            issue_s(0);
        }
    }
    for (int it = 0; it < n; ++it) {
        // (A) the next tile's scores run under this tile's softmax
        if (it + 1 < n) {
            cp_wait<1>();  // tiles <= it + 1 landed (it + 2 may be in flight)
            fence_proxy_async();
            fence_before();
            __syncthreads();
            if (tid == 0) {
                fence_after();
                issue_s(it + 1);
            }
        }
        // (B) this tile's scores
        wait(&bar_s[it & 1], (uint32_t)((it >> 1) & 1));
        fence_after();
        float sc[KH];
        {
            const uint32_t tS = tmem + t_lane + (uint32_t)((it & 1) * KT + KH * half);
            uint32_t r_[KH / 16][16];
#pragma unroll
            for (int q = 0; q < KH / 16; ++q) tmem_ld16_issue(tS + 16 * q, r_[q]);
#pragma unroll
            for (int q = 0; q < KH / 16; ++q) tmem_ld_wait(r_[q]);
#pragma unroll
            for (int q = 0; q < KH / 16; ++q)
#pragma unroll
                for (int c = 0; c < 16; ++c) sc[16 * q + c] = __uint_as_float(r_[q][c]);
        }
        // (C) online softmax, lazy reference max (moves only by more than 2^8); the row's
        // tile max from all its parts (the warps of quadrant w % 4 meet at named barrier 1 + w % 4)
        float mx = -INFINITY;
        const int k0 = it * KT + KH * half;
#pragma unroll
        for (int c = 0; c < KH; ++c) {
            sc[c] = (k0 + c < lim) ? sc[c] * a.scale_log2 : -INFINITY;
            mx = fmaxf(mx, sc[c]);
        }
        xch_s[half][v] = mx;
        asm volatile("bar.sync %0, %1;" ::"r"(1 + (warp & 3)), "n"(32 * NSPLIT) : "memory");
#pragma unroll
        for (int q = 0; q < NSPLIT; ++q) mx = fmaxf(mx, xch_s[q][v]);
        asm volatile("bar.sync %0, %1;" ::"r"(1 + (warp & 3)), "n"(32 * NSPLIT) : "memory");  // all read first
        const float m_new = (mx > m_run + 8.f) ? mx : m_run;
        const float alpha = (m_new == m_run) ? 1.f : ((m_run == -INFINITY) ? 0.f : exp2f(m_run - m_new));
        float sum = 0.f;  // this half's share; the halves' running sums are added at the end
#pragma unroll
        for (int c = 0; c < KH; ++c) {
            sc[c] = (sc[c] == -INFINITY) ? 0.f : exp2f(sc[c] - m_new);
            sum += sc[c];
        }
        l_run = l_run * alpha + sum;
        m_run = m_new;
        // (D) the previous P.V has released P, O and ring stage (it - 1) % RING
        if (it > 0) {
            wait(bar_o, (uint32_t)((it - 1) & 1));
            fence_after();
        }
#pragma unroll
        for (int ch = 0; ch < KH / 8; ++ch) {  // this part's 16-byte chunks of row v
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float x0 = sc[8 * ch + 2 * e], x1 = sc[8 * ch + 2 * e + 1];
                hi[e] = pack2_bf16(x0, x1);
                lo[e] = pack2_bf16(x0 - __uint_as_float(hi[e] << 16), x1 - __uint_as_float(hi[e] & 0xFFFF0000u));
            }
            *reinterpret_cast<uint4*>(sm + P_OFF + swz(v, (KH / 8) * half + ch)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<uint4*>(sm + P_OFF + QM * 128 + swz(v, (KH / 8) * half + ch)) =
                make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
        // rescale the running O when the reference max moved (warp-collective TMEM access)
        if (it > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
            for (int c = 0; c < OH; c += 16) {
                float o[16];
                tmem_ld16(tO + c, o);
#pragma unroll
                for (int e = 0; e < 16; ++e) o[e] *= alpha;
                tmem_st16(tO + c, o);
            }
        }
        // (E) O += P_hi V + P_lo V
        fence_proxy_async();
        fence_before();
        __syncthreads();
        if (tid == 0) {
            fence_after();
            const uint32_t ph = sb + P_OFF, pl = sb + P_OFF + QM * 128;
            const uint32_t vb = sb + V_OFF + (it % RING) * 2 * KV_REG;
#pragma unroll
            for (int kk = 0; kk < KT / 16; ++kk)
                umma_bf16(tmem + 128, sw128_desc(ph + kk * 32), sw128_desc(vb + kk * 2048, KV_REG, 1024), ID_O,
                          (it > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
            for (int kk = 0; kk < KT / 16; ++kk)
                umma_bf16(tmem + 128, sw128_desc(pl + kk * 32), sw128_desc(vb + kk * 2048, KV_REG, 1024), ID_O, 1u);
            umma_commit(bar_o);
        }
        // (F) K/V of tile it + 3 into the stage of tile it - 1 (its S and P.V have completed)
        load_tile(it + 3);
    }
    cp_wait<0>();
    if (n > 0) {
        wait(bar_o, (uint32_t)((n - 1) & 1));
        fence_after();
    }
    xch_s[half][v] = l_run;
    __syncthreads();
    if (n > 0) {
        __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out);
        float l = 0.f;
#pragma unroll
        for (int q = 0; q < NSPLIT; ++q) l += xch_s[q][v];
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const bool live = okw && v < nv && lim > 0;
        __nv_bfloat16* dst =
            live ? out + (size_t)(r0 + v / g) * p.H * HD + (size_t)(kvh * g + v % g) * HD + OH * half : nullptr;
#pragma unroll 1
        for (int c = 0; c < OH; c += 16) {
            float o[16];
            tmem_ld16(tO + c, o);
            if (dst) {
#pragma unroll
                for (int e = 0; e < 16; e += 2)
                    *reinterpret_cast<__nv_bfloat162*>(dst + c + e) = __floats2bfloat162_rn(o[e] * inv, o[e + 1] * inv);
            }
        }
    }
    fence_before();
    __syncthreads();
    if (warp == 0) {
        fence_after();
        tmem_dealloc(tmem, 256);
    }
}

}  // namespace

// Causal prefill attention on tcgen05: head_dim 128, group_rows * (H / H_kv) == 128, and the
// rows of every query group in one sequence (sequence-major rows with seq_div a multiple of
// group_rows, or seq_div == 0 with row_seq constant over each group, as in a prefill chunk).
// Returns false (nothing launched) otherwise.
bool attention_prefill_tc(const Launch& L, const AttnParams& p) {
    if (p.rows <= 0) return true;
    if (p.hd != HD || p.H % p.Hkv || p.seq_len) return false;
    if (p.seq_div > 0 && p.seq_div % p.group_rows) return false;
    const int g = p.H / p.Hkv;
    if (g * p.group_rows != QM) return false;
    PfArgs a;
    a.p = p;
    a.g = g;
    a.scale_log2 = 1.4426950408889634f / sqrtf((float)HD);
    a.err = L.err;
    static bool attr = false;
    if (!attr) {
        if (cudaFuncSetAttribute(attn_prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM) !=
            cudaSuccess)
            return false;
        attr = true;
    }
    const int n_groups = (p.rows + p.group_rows - 1) / p.group_rows;
    launch_k(L, attn_prefill_tc_kernel, dim3(n_groups, p.Hkv), dim3(NT), (size_t)SMEM, 1, a);
    return true;
}

}  // namespace dfl
