// Tensor-core GEMM for bf16 operands on sm_103a (tcgen05 + TMA + TMEM):
//
//     C[M, N] (fp32, row stride ldc)  =|+=  A[M, K] (bf16) . W[N, K]^T (bf16)
//
// The weight matrix is the MMA's A operand: each CTA owns a 128-row slab of W
// (128 output features) and one range of K; the activations (the M token rows,
// at most 256 per tile) are the B operand, so the accumulator D[128, M_tile]
// lives in TMEM with one output feature per lane.  This "swap" keeps the
// tensor cores usable when M is only a block of 16 tokens: the work is the
// weight stream, and every weight byte is read from HBM once.
//
// Warp roles (192 threads): warp 0 issues TMA loads (one elected lane), warp 1
// allocates TMEM and issues tcgen05.mma (one elected lane), warps 2-5 drain the
// accumulator (tcgen05.ld; warp w reads TMEM lanes 32*(w%4) .. +31).  A ring of
// STAGES shared-memory stages (128-byte swizzled, as TMA writes them and as
// the UMMA descriptors read them) is guarded by full/empty mbarriers.
//
// Split-K: when the N tiles alone cannot fill the GPU, K is cut into `splits`
// (<= 8) contiguous ranges whose CTAs form one thread-block cluster.  Each CTA
// parks its fp32 partial tile in its own shared memory; after a cluster
// barrier, CTA r sums columns [r*MT/S, (r+1)*MT/S) of the tile over the peers'
// shared memory (distributed shared memory), always in rank order, so the
// result does not depend on scheduling, and applies the epilogue.
//
// Programmatic dependent launch: the producer fills the first STAGES weight
// tiles before waiting for the previous kernel (weights never depend on it),
// so the weight stream of this GEMM overlaps the tail of the kernel before.
//
// Every wait on an mbarrier is bounded; a wait that runs out sets ERR_TIMEOUT
// in the error word, and the CTA still reaches its cluster barriers, releases
// its TMEM and returns.
#include <cuda.h>
#include <string.h>

#include <algorithm>

#include <mutex>
#include <unordered_map>

#include "launch.h"
#include "tcgen05.cuh"

namespace dfl {

namespace {

constexpr int BN = 128;          // weight rows per tile = UMMA M
constexpr int BK = 64;           // K per stage: one 128-byte swizzle row of bf16
constexpr int UMMA_K = 16;
constexpr int THREADS = 192;
using namespace tc;

struct QkvEpi {
    int q_tiles, n_kv;
    const float* q_norm;
    const float* k_norm;
    const float2* rope;  // [max_pos][64]
    int max_pos;
    __nv_bfloat16* q_out;
    __nv_bfloat16* Kc;
    __nv_bfloat16* Vc;
    KVLayout kv;
    const int* page_table;
    const int* row_seq;
    const int* row_pos;
    int layer_tiles;          // tiles of one layer (q_tiles + 2 n_kv)
    long long layer_stride;   // cache elements between layers
    int norm_stride;          // k_norm floats between layers
};

struct TcArgs {
    float* C;
    int ldc, M, N, K;
    int accumulate;
    int splits;
    int kb_per_split;
    int n_tiles;
    uint32_t* err;
    // A operand normalised on the fly (NORM_A): bf16(x * rstd[m] * norm_w[k]), with
    // rstd[m] = 1/sqrt(sum_t ss_in[t][m] / K + eps) from per-tile sums of squares
    const float* norm_w;
    const float* ss_in;
    int ss_tiles, ss_ld;
    float eps;
    // epilogue: 0 = fp32 C (=|+=); 1 = SwiGLU: tile rows 16g + i (i < 8) are the gate and
    // rows 16g + 8 + i the up projection of feature 64*tile + 8g + i, written as bf16
    // silu(gate) * up to out[m * ldo + f]
    int epi;
    void* out;
    int ldo;
    // epilogue 0: per-(tile, row) sum of squares of the final C values (or null)
    float* ss_out;
    // epilogue 2 (argmax): keys[m] = max over n of argmax_key(C[m][n], n) (C also written when set)
    unsigned long long* keys;
    // epilogue 3 (q/k/v of head_dim 128: one head per tile): tiles [0, q_tiles) are query heads,
    // then n_kv key heads, then n_kv value heads; per-head RMSNorm of q (q_norm) and k (k_norm),
    // RoPE at row_pos[m], q to q_out [M, q_tiles*128], k and v into the paged cache at
    // (row_seq[m], row_pos[m]); rows with row_seq < 0 are skipped
    QkvEpi qkv;
};

template <int MT, int STAGES, bool NORM_A>
struct Smem {
    static constexpr int W_BYTES = BN * BK * 2;             // 16 KB weight tile
    static constexpr int X_BYTES = MT * BK * 2;             // bf16 activation tile (MMA operand)
    static constexpr int XRAW_BYTES = NORM_A ? MT * BK * 4 : 0;  // fp32 residual tile (NORM_A)
    static constexpr int STAGE_BYTES = W_BYTES + X_BYTES + XRAW_BYTES;
    static constexpr int NW_OFF = STAGES * STAGE_BYTES;           // NORM_A: norm weights of each stage's K slice
    static constexpr int BAR_OFF = NW_OFF + (NORM_A ? STAGES * BK * 4 : 0);
    static constexpr int NBAR = 2 * STAGES + 1 + (NORM_A ? 2 * STAGES : 0);
    static constexpr int TOTAL = BAR_OFF + NBAR * 8 + 16 + 64 * 4 + 128 * 4 + 1024;  // + rstd, partial sums, alignment
};

// Sync of the four epilogue warps (warps 2..5) only.
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

template <int MT, int STAGES, bool NORM_A>
__global__ void __launch_bounds__(THREADS, (MT <= 64 ? 2 : 1)) tc_gemm_kernel(const __grid_constant__ CUtensorMap tmW,
                                                          const __grid_constant__ CUtensorMap tmX, TcArgs a) {
    using S = Smem<MT, STAGES, NORM_A>;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment for the swizzled tiles
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::BAR_OFF);
    uint64_t* empty = full + STAGES;
    uint64_t* accf = empty + STAGES;
    uint64_t* xraw = accf + 1;          // NORM_A: raw fp32 tile landed
    uint64_t* conv = xraw + STAGES;     // NORM_A: bf16 operand written by the epilogue warps
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + S::BAR_OFF + S::NBAR * 8);
    float* rstd_s = reinterpret_cast<float*>(tmem_slot + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // token tiles run fastest: the token tiles of one weight tile run together and share
    // its L2 copy (the weight stream is read from DRAM once)
    const int mt = blockIdx.x, nt = blockIdx.y, split = blockIdx.z;
    const int n0 = nt * BN, m0 = mt * MT;
    const int KB = (a.K + BK - 1) / BK;
    const int kb0 = split * a.kb_per_split;
    const int kb1 = min(KB, kb0 + a.kb_per_split);
    const int nkb = kb1 - kb0;
    constexpr uint32_t TMEM_COLS = MT < 32 ? 32 : MT;

    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmW);
        prefetch_tmap(&tmX);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
            if (NORM_A) {
                mbar_init(&xraw[s], 1);
                mbar_init(&conv[s], 128);
            }
        }
        mbar_init(accf, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *tmem_slot;

    pdl_trigger();  // the next kernel may start its own prologue now

    bool ok = true;
    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pw = policy_evict_first(), px = policy_evict_last();
            constexpr uint32_t FULL_TX = NORM_A ? S::W_BYTES : S::W_BYTES + S::X_BYTES;
            // weights of the first stages do not depend on the previous kernel
            const int pre = nkb < STAGES ? nkb : STAGES;
            for (int i = 0; i < pre; ++i) {
                mbar_arrive_expect_tx(&full[i], FULL_TX);
                tma_load_2d(smem + i * S::STAGE_BYTES, &tmW, &full[i], (kb0 + i) * BK, n0, pw);
            }
            pdl_wait();
            for (int i = 0; i < pre; ++i) {
                uint8_t* st = smem + i * S::STAGE_BYTES;
                if (NORM_A) {
                    const int kc = (kb0 + i) * BK;
                    const uint32_t nwb = (uint32_t)min(BK, a.K - kc) * 4u;
                    mbar_arrive_expect_tx(&xraw[i], S::XRAW_BYTES + nwb);
                    tma_load_2d(st + S::W_BYTES + S::X_BYTES, &tmX, &xraw[i], kc, m0, px);
                    bulk_load(smem + S::NW_OFF + i * BK * 4, a.norm_w + kc, nwb, &xraw[i]);
                } else {
                    tma_load_2d(st + S::W_BYTES, &tmX, &full[i], (kb0 + i) * BK, m0, px);
                }
            }
            for (int i = pre; i < nkb; ++i) {
                const int s = i % STAGES;
                if (!mbar_wait(&empty[s], ((i / STAGES) + 1) & 1, a.err)) {
                    ok = false;
                    break;
                }
                uint8_t* st = smem + s * S::STAGE_BYTES;
                const int kc = (kb0 + i) * BK;
                mbar_arrive_expect_tx(&full[s], FULL_TX);
                tma_load_2d(st, &tmW, &full[s], kc, n0, pw);
                if (NORM_A) {
                    const uint32_t nwb = (uint32_t)min(BK, a.K - kc) * 4u;
                    mbar_arrive_expect_tx(&xraw[s], S::XRAW_BYTES + nwb);
                    tma_load_2d(st + S::W_BYTES + S::X_BYTES, &tmX, &xraw[s], kc, m0, px);
                    bulk_load(smem + S::NW_OFF + s * BK * 4, a.norm_w + kc, nwb, &xraw[s]);
                } else {
                    tma_load_2d(st + S::W_BYTES, &tmX, &full[s], kc, m0, px);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16(BN, MT);
            for (int i = 0; i < nkb; ++i) {
                const int s = i % STAGES;
                if (!mbar_wait(&full[s], (i / STAGES) & 1, a.err)) {
                    ok = false;
                    break;
                }
                if (NORM_A && !mbar_wait(&conv[s], (i / STAGES) & 1, a.err)) {
                    ok = false;
                    break;
                }
                fence_after();
                const uint32_t sw = smem_u32(smem + s * S::STAGE_BYTES);
                const uint32_t sx = sw + S::W_BYTES;
#pragma unroll
                for (int kk = 0; kk < BK / UMMA_K; ++kk)
                    umma_bf16(tmem, sw128_desc(sw + kk * UMMA_K * 2), sw128_desc(sx + kk * UMMA_K * 2), idesc,
                              (i > 0 || kk > 0) ? 1u : 0u);
                umma_commit(&empty[s]);
            }
            umma_commit(accf);  // fires once every MMA issued above has completed
        }
    } else if (NORM_A) {
        // epilogue warps convert each raw fp32 tile into the normalised bf16 operand
        pdl_wait();
        const int e = threadIdx.x - 64;  // 0..127
        {
            // rstd of the MT rows: thread (part, m) sums tiles part, part + P, ... (loads issued
            // together), then the P part sums are added in a fixed order
            constexpr int P = 128 / MT;
            float* psum = rstd_s + 64;  // [P][MT]
            const int m = e % MT, part = e / MT;
            float acc = 0.f;
            if (m0 + m < a.M) {
                float v[8];
                for (int t0 = part; t0 < a.ss_tiles; t0 += 8 * P) {
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int t = t0 + u * P;
                        v[u] = t < a.ss_tiles ? __ldcg(a.ss_in + (size_t)t * a.ss_ld + m0 + m) : 0.f;
                    }
#pragma unroll
                    for (int u = 0; u < 8; ++u) acc += v[u];
                }
            }
            psum[part * MT + m] = acc;
            epi_sync();
            if (e < MT) {
                float ss = 0.f;
#pragma unroll
                for (int p2 = 0; p2 < P; ++p2) ss += psum[p2 * MT + e];
                rstd_s[e] = rsqrtf(ss / (float)a.K + a.eps);
            }
            epi_sync();
        }
        for (int i = 0; i < nkb; ++i) {
            const int s = i % STAGES;
            uint8_t* st = smem + s * S::STAGE_BYTES;
            const int kc = (kb0 + i) * BK;
            const int c = e & 7;
            const int k = kc + 8 * c;
            // the raw tile and the stage's norm weights land together (one barrier)
            if (!mbar_wait(&xraw[s], (i / STAGES) & 1, a.err)) ok = false;
            const float* nw = reinterpret_cast<const float*>(smem + S::NW_OFF + s * BK * 4) + 8 * c;
            float w8[8];
            if (k + 8 <= a.K) {
                const float4 w0 = reinterpret_cast<const float4*>(nw)[0];
                const float4 w1 = reinterpret_cast<const float4*>(nw)[1];
                w8[0] = w0.x; w8[1] = w0.y; w8[2] = w0.z; w8[3] = w0.w;
                w8[4] = w1.x; w8[5] = w1.y; w8[6] = w1.z; w8[7] = w1.w;
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) w8[j] = (k + j < a.K) ? nw[j] : 0.f;  // past K: not loaded
            }
            const float* xr = reinterpret_cast<const float*>(st + S::W_BYTES + S::X_BYTES);
            uint8_t* xb = st + S::W_BYTES;
            // 16-byte output chunks: row m, k-chunk c (8 elements); swizzle chunk ^ (m & 7)
            for (int ch = e; ch < MT * 8; ch += 128) {
                const int m = ch >> 3;
                const float4 x0 = *reinterpret_cast<const float4*>(xr + m * BK + 8 * c);
                const float4 x1 = *reinterpret_cast<const float4*>(xr + m * BK + 8 * c + 4);
                const float r = rstd_s[m];
                uint4 o;
                o.x = pack2_bf16(x0.x * r * w8[0], x0.y * r * w8[1]);
                o.y = pack2_bf16(x0.z * r * w8[2], x0.w * r * w8[3]);
                o.z = pack2_bf16(x1.x * r * w8[4], x1.y * r * w8[5]);
                o.w = pack2_bf16(x1.z * r * w8[6], x1.w * r * w8[7]);
                *reinterpret_cast<uint4*>(xb + m * 128 + ((c ^ (m & 7)) << 4)) = o;
            }
            // generic-proxy writes must be visible to the tensor core's async proxy
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            mbar_arrive(&conv[s]);
        }
    }
    __syncwarp();
    pdl_wait();  // every thread: the previous kernel's outputs (C when accumulating) are visible

    const int q = warp & 3;
    const int row = 32 * q + lane;  // feature within the tile
    const int n = n0 + row;
    float* part = reinterpret_cast<float*>(smem);                  // [MT][BN] partial tile (cluster split-K)
    float* xch = a.splits > 1 ? part + MT * BN : part;             // [MT][BN] final values (SwiGLU exchange)
    float* ssw = xch + ((a.epi == 1 || a.epi == 3) ? MT * BN : 0);  // [4][MT] per-warp sums of squares
    unsigned long long* wkey = reinterpret_cast<unsigned long long*>(ssw + 4 * MT);  // [4][MT] argmax keys
    const bool epi_warp = warp >= 2;
    uint32_t okw = 0;
    if (epi_warp) {
        if (lane == 0) okw = mbar_wait(accf, 0, a.err) ? 1u : 0u;
        ok = __shfl_sync(0xffffffffu, okw, 0) != 0;
        fence_after();
    }

    // Kernel arguments used per token, hoisted into registers once.
    const int epi = a.epi;
    float* const Cp = a.C;
    const size_t ldc = (size_t)a.ldc;
    const bool accum = a.accumulate != 0;
    const bool has_ss = a.ss_out != nullptr;
    const bool n_ok = n < a.N;
    const int m_left = a.M - m0;  // tokens j < m_left of this tile are real rows

    // Final value of (token j, this row) -> C / exchange tile / sum of squares / argmax key.
    auto finish = [=](int j, float v) {
        if (epi == 0) {
            float f = 0.f;
            if (n_ok && j < m_left) {
                float* dst = Cp + (size_t)(m0 + j) * ldc + n;
                f = accum ? (*dst + v) : v;
                *dst = f;
            }
            if (has_ss) {
                const float sq = warp_sum(f * f);
                if (lane == 0) ssw[q * MT + j] = sq;
            }
        } else if (epi == 1 || epi == 3) {
            xch[j * BN + row] = v;
        } else {
            unsigned long long key = 0ull;
            if (n_ok && j < m_left) {
                if (Cp) Cp[(size_t)(m0 + j) * ldc + n] = v;
                key = argmax_key(v, (uint32_t)n);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const unsigned long long t = __shfl_xor_sync(0xffffffffu, key, o);
                key = t > key ? t : key;
            }
            if (lane == 0) wkey[q * MT + j] = key;
        }
    };

    if (a.splits == 1) {
        if (epi_warp) {
            const uint32_t tbase = tmem + ((uint32_t)(32 * q) << 16);
            float v[16];
            // Groups of 16 accumulator columns, kept rolled (an unrolled loop would hold
            // MT copies of the epilogue code); one specialised loop per epilogue kind.
#pragma unroll 1
            for (int c = 0; c < MT; c += 16) {
                if (ok) tmem_ld16(tbase + c, v);
                else {
#pragma unroll
                    for (int j = 0; j < 16; ++j) v[j] = 0.f;
                }
                if (epi == 0 && !has_ss) {
                    float* dst = Cp + (size_t)(m0 + c) * ldc + n;
                    const int lim = n_ok ? min(16, m_left - c) : 0;
                    if (accum) {
                        float old[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) old[j] = j < lim ? dst[j * ldc] : 0.f;
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            if (j < lim) dst[j * ldc] = old[j] + v[j];
                    } else {
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            if (j < lim) dst[j * ldc] = v[j];
                    }
                } else if (epi == 0) {
                    // C update plus the per-token sum of squares over the tile's 128 rows
                    float* dst = Cp + (size_t)(m0 + c) * ldc + n;
                    const int lim = n_ok ? min(16, m_left - c) : 0;
                    float f[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) f[j] = (accum && j < lim) ? dst[j * ldc] : 0.f;
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        f[j] = j < lim ? f[j] + v[j] : 0.f;
                        if (j < lim) dst[j * ldc] = f[j];
                        f[j] *= f[j];
                    }
                    const float sq = transpose_reduce16(f, lane, [](float x, float y) { return x + y; });
                    if (!(lane & 1)) ssw[q * MT + c + (lane >> 1)] = sq;
                } else if (epi == 1 || epi == 3) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) xch[(c + j) * BN + row] = v[j];
                } else {
                    // row argmax keys: the best (value, index) of each token over the tile's rows
                    const int lim = n_ok ? min(16, m_left - c) : 0;
                    unsigned long long k[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        k[j] = j < lim ? argmax_key(v[j], (uint32_t)n) : 0ull;
                        if (Cp && j < lim) Cp[(size_t)(m0 + c + j) * ldc + n] = v[j];
                    }
                    const unsigned long long best = transpose_reduce16(
                        k, lane, [](unsigned long long x, unsigned long long y) { return x > y ? x : y; });
                    if (!(lane & 1)) wkey[q * MT + c + (lane >> 1)] = best;
                }
            }
        }
    } else {
        // ---- cluster split-K: rank r reduces its slice of columns over all ranks, in rank order
        if (epi_warp) {
            const uint32_t tbase = tmem + ((uint32_t)(32 * q) << 16);
            float v[16];
#pragma unroll 1
            for (int c = 0; c < MT; c += 16) {  // rolled: an unrolled body is MT copies of the epilogue code
                if (ok) tmem_ld16(tbase + c, v);
                else {
#pragma unroll
                    for (int j = 0; j < 16; ++j) v[j] = 0.f;
                }
#pragma unroll
                for (int j = 0; j < 16; ++j) part[(c + j) * BN + row] = v[j];
            }
        }
        cluster_sync();
        const uint32_t rank = cluster_rank();
        const int per = (MT + a.splits - 1) / a.splits;
        const int j0 = (int)rank * per;
        const int j1 = min(MT, j0 + per);
        if (epi_warp) {
            for (int j = j0; j < j1; ++j) {
                float vals[8];
#pragma unroll
                for (int r = 0; r < 8; ++r) vals[r] = (r < a.splits) ? ld_peer(part + j * BN + row, (uint32_t)r) : 0.f;
                float acc = 0.f;
#pragma unroll
                for (int r = 0; r < 8; ++r)
                    if (r < a.splits) acc += vals[r];
                finish(j, acc);
            }
        }
        cluster_sync();  // peers keep their shared memory until every slice is read
    }

    // ---- per-row sums of squares (epilogue 0), SwiGLU (1) and argmax (2) need all 128 rows
    if (epi_warp && (a.ss_out || a.epi != 0)) {
        epi_sync();
        int j0 = 0, j1 = MT;
        if (a.splits > 1) {
            const int per = (MT + a.splits - 1) / a.splits;
            j0 = (int)cluster_rank() * per;
            j1 = min(MT, j0 + per);
        }
        // one token per epilogue thread, 128 at a time (tiles of 256 tokens take two passes)
        if (a.ss_out) {
            for (int e = threadIdx.x - 64; e < j1 - j0; e += 128) {
                const int j = j0 + e, m = m0 + j;
                if (m < a.M) a.ss_out[(size_t)nt * a.ss_ld + m] = ((ssw[j] + ssw[MT + j]) + ssw[2 * MT + j]) + ssw[3 * MT + j];
            }
        }
        if (a.epi == 2) {
            for (int e = threadIdx.x - 64; e < j1 - j0; e += 128) {
                const int j = j0 + e, m = m0 + j;
                unsigned long long best = wkey[j];
#pragma unroll
                for (int w2 = 1; w2 < 4; ++w2) best = wkey[w2 * MT + j] > best ? wkey[w2 * MT + j] : best;
                if (m < a.M) atomicMax(a.keys + m, best);
            }
        }
        if (a.epi == 3) {
            const QkvEpi& Q = a.qkv;
            const int layer = nt / Q.layer_tiles, lt = nt - layer * Q.layer_tiles;
            const int kind = lt < Q.q_tiles ? 0 : (lt < Q.q_tiles + Q.n_kv ? 1 : 2);  // q / k / v head
            const int head = kind == 0 ? lt : (kind == 1 ? lt - Q.q_tiles : lt - Q.q_tiles - Q.n_kv);
            const float* nw =
                kind == 0 ? Q.q_norm : (kind == 1 && Q.k_norm ? Q.k_norm + (size_t)layer * Q.norm_stride : nullptr);
            if (nw) {
                // per-head RMSNorm over the tile's 128 rows (each thread rescales only its own row)
                for (int j = j0; j < j1; ++j) {
                    const float x = xch[j * BN + row];
                    const float sq = warp_sum(x * x);
                    if (lane == 0) ssw[q * MT + j] = sq;
                }
                epi_sync();
                const float w = nw[row];
                for (int j = j0; j < j1; ++j) {
                    const float ss = ((ssw[j] + ssw[MT + j]) + ssw[2 * MT + j]) + ssw[3 * MT + j];
                    xch[j * BN + row] = xch[j * BN + row] * rsqrtf(ss / (float)BN + a.eps) * w;
                }
            }
            if (kind < 2) epi_sync();  // RoPE reads the partner row
            for (int j = j0; j < j1; ++j) {
                const int m = m0 + j;
                if (m >= a.M) break;
                const int seq = Q.row_seq[m], pos = Q.row_pos[m];
                if (seq < 0) continue;
                if (pos < 0 || pos >= Q.max_pos) {
                    if (row == 0 && a.err) atomicOr(a.err, ERR_POSITION_RANGE);
                    continue;
                }
                float val = xch[j * BN + row];
                if (kind < 2) {
                    const float partner = xch[j * BN + (row ^ 64)];
                    const float2 cs = Q.rope[(size_t)pos * 64 + (row & 63)];
                    val = row < 64 ? val * cs.x - partner * cs.y : val * cs.x + partner * cs.y;
                }
                const __nv_bfloat16 o = __float2bfloat16_rn(val);
                if (kind == 0) {
                    Q.q_out[(size_t)m * Q.q_tiles * BN + (size_t)head * BN + row] = o;
                } else {
                    __nv_bfloat16* base = (kind == 1 ? Q.Kc : Q.Vc) + (size_t)layer * Q.layer_stride;
                    base[kv_offset(Q.kv, Q.page_table, seq, pos, head) + row] = o;
                }
            }
        }
        if (a.epi == 1) {
            // thread e: feature r = e % 64 of tokens j0 + e / 64, +2, ...; the tile holds gate and
            // up rows in alternating groups of eight (gate of feature r at row gr, its up at gr + 8);
            // four tokens per iteration as independent chains (one warp per scheduler here)
            const int e = threadIdx.x - 64;
            const int r = e & 63;
            const int gr = ((r >> 3) << 4) | (r & 7);
            const int f = 64 * nt + r;
            __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.out) + f;
            const size_t ldo = (size_t)a.ldo;
            const int jend = min(j1, a.M - m0);
            // silu(g) * u with the fast exponential and division (a gate below about -88 gives
            // an infinite denominator and a zero result, the function's limit)
            auto swiglu = [](float gte, float up) { return __fdividef(gte, 1.f + __expf(-gte)) * up; };
            if (n0 + r < a.N) {
                int j = j0 + (e >> 6);
                for (; j + 6 < jend; j += 8) {
                    float gv[4], uv[4];
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        gv[t] = xch[(j + 2 * t) * BN + gr];
                        uv[t] = xch[(j + 2 * t) * BN + gr + 8];
                    }
#pragma unroll
                    for (int t = 0; t < 4; ++t)
                        out[(size_t)(m0 + j + 2 * t) * ldo] = __float2bfloat16_rn(swiglu(gv[t], uv[t]));
                }
                for (; j < jend; j += 2)
                    out[(size_t)(m0 + j) * ldo] =
                        __float2bfloat16_rn(swiglu(xch[j * BN + gr], xch[j * BN + gr + 8]));
            }
        }
    }

    fence_before();
    __syncthreads();
    if (warp == 1) {
        fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ------------------------------------------------------------------ host side
// Split count (cluster size): the largest power of two that keeps the grid within
// one wave of `slots` CTAs.  The cluster reduction of the [MT x 128] fp32 partial
// tile grows with MT, so wider tiles split less: up to 8 ways for tiles of <= 32
// tokens (>= 4 K blocks per split), 4 ways for 64 (>= 4) and 128 (>= 48 K blocks
// per split, i.e. long K only), never for 256.
int choose_splits(int tiles, int kb, int slots, int mt) {
    if (mt >= 256) return 1;
    const int cap = mt <= 32 ? 8 : 4;
    const int min_kb = mt <= 64 ? 4 : 48;
    int s = 1;
    while (s < cap && (long long)tiles * (2 * s) <= slots && kb / (2 * s) >= min_kb) s *= 2;
    return s;
}

template <int MT, int STAGES, bool NORM_A>
bool launch_tc(const Launch& L, const CUtensorMap& mw, const CUtensorMap& mx, TcArgs a, int m_tiles) {
    using S = Smem<MT, STAGES, NORM_A>;
    static bool attr = false;
    if (!attr) {
        if (cudaFuncSetAttribute(tc_gemm_kernel<MT, STAGES, NORM_A>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 S::TOTAL) != cudaSuccess)
            return false;
        cudaFuncSetAttribute(tc_gemm_kernel<MT, STAGES, NORM_A>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
        attr = true;
    }
    const int KB = (a.K + BK - 1) / BK;
    const int cta_per_sm = S::TOTAL <= 113 * 1024 ? 2 : 1;
    int splits = choose_splits(a.n_tiles * m_tiles, KB, sm_count() * cta_per_sm, MT);
    // the epilogue reuses the stage memory: partials (split-K) + exchange (SwiGLU) + row sums
    auto fits = [&](int sp) {
        const size_t need = (sp > 1 ? (size_t)MT * BN * 4 : 0) +
                            ((a.epi == 1 || a.epi == 3) ? (size_t)MT * BN * 4 : 0) + 16 * MT + 32 * MT;
        return need <= (size_t)STAGES * S::STAGE_BYTES;
    };
    if (!fits(splits)) splits = 1;
    if (!fits(1)) return false;
    a.kb_per_split = (KB + splits - 1) / splits;
    a.splits = (KB + a.kb_per_split - 1) / a.kb_per_split;
    dim3 grid(m_tiles, a.n_tiles, a.splits);
    launch_k(L, tc_gemm_kernel<MT, STAGES, NORM_A>, grid, dim3(THREADS), (size_t)S::TOTAL, a.splits, mw, mx, a);
    return true;
}

}  // namespace

namespace tc {

namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

struct MapKey {
    const void* ptr;
    long long rows, cols, ld;
    int box_rows, f32;
    bool operator==(const MapKey& o) const {
        return ptr == o.ptr && rows == o.rows && cols == o.cols && ld == o.ld && box_rows == o.box_rows && f32 == o.f32;
    }
};
struct MapKeyHash {
    size_t operator()(const MapKey& k) const {
        size_t h = std::hash<const void*>()(k.ptr);
        h ^= std::hash<long long>()(k.rows * 1000003LL + k.cols) + 0x9e3779b97f4a7c15ull + (h << 6) + (h >> 2);
        h ^= std::hash<long long>()(k.ld * 131 + k.box_rows * 2 + k.f32) + 0x9e3779b97f4a7c15ull + (h << 6) + (h >> 2);
        return h;
    }
};
}  // namespace

bool make_map(CUtensorMap* out, const void* ptr, long long rows, long long cols, long long ld, int box_rows,
              bool f32) {
    static std::mutex mu;
    static std::unordered_map<MapKey, CUtensorMap, MapKeyHash> cache;
    const MapKey key{ptr, rows, cols, ld, box_rows, f32 ? 1 : 0};
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) {
        *out = it->second;
        return true;
    }
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const int esz = f32 ? 4 : 2;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ld * esz};
    cuuint32_t box[2] = {64u, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUtensorMap m;
    CUresult r = fn(&m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                    const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    f32 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
    if (cache.size() > 65536) cache.clear();
    cache.emplace(key, m);
    *out = m;
    return true;
}

int sm_count() {
    static int n = 0;
    if (!n) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n <= 0) n = 148;
    }
    return n;
}

}  // namespace tc

// bf16 GEMM on the tensor cores.  Returns false when a tensor map cannot be
// built (the caller reports the error); nothing is launched in that case.
bool gemm_tc(const Launch& L, const bf16* A, int lda, int a_rows, const bf16* W, int M, int N, int K, float* C,
             int ldc, bool accumulate, const GemmEpi* ep) {
    static const GemmEpi none;
    if (!ep) ep = &none;
    const bool norm_a = ep->x_f32 != nullptr;
    int MT;
    if (M <= 16) MT = 16;
    else if (M <= 32) MT = 32;
    else if (M <= 64) MT = 64;
    else if (M <= 128) MT = 128;
    else MT = 256;
    if (norm_a && MT > 32) return false;  // the fused norm serves blocks of at most 32 rows
    if (!norm_a) {
        // Narrower token tiles while the grid is under one wave and the narrower grid still
        // fits in one (tiles of <= 64 tokens run two CTAs per SM, so one CTA's epilogue
        // overlaps the other's main loop).
        const int n_tiles = (N + BN - 1) / BN, sms = sm_count();
        auto tiles = [&](int mt) { return n_tiles * ((M + mt - 1) / mt); };
        auto slots = [&](int mt) { return sms * (mt <= 64 ? 2 : 1); };
        while (MT > 64 && tiles(MT) < slots(MT) && tiles(MT / 2) <= slots(MT / 2)) MT /= 2;
    }
    CUtensorMap mw, mx;
    if (!make_map(&mw, W, N, K, K, BN)) return false;
    if (norm_a) {
        // the norm weights reach shared memory by bulk copies of each stage's K slice
        if ((reinterpret_cast<uintptr_t>(ep->norm_w) & 15) != 0) return false;
        if (!make_map(&mx, ep->x_f32, a_rows, K, ep->ldx, MT, true)) return false;
    } else if (!make_map(&mx, A, a_rows, K, lda, MT)) {
        return false;
    }
    TcArgs a;
    memset(&a, 0, sizeof a);
    a.C = C;
    a.ldc = ldc;
    a.M = M;
    a.N = N;
    a.K = K;
    a.accumulate = accumulate ? 1 : 0;
    a.n_tiles = (N + BN - 1) / BN;
    a.err = L.err;
    a.splits = 1;
    a.norm_w = ep->norm_w;
    a.ss_in = ep->ss_in;
    a.ss_tiles = ep->ss_tiles;
    a.ss_ld = ep->ss_ld;
    a.eps = ep->eps;
    a.epi = ep->epi;
    a.out = ep->out;
    a.ldo = ep->ldo;
    a.ss_out = ep->ss_out;
    a.keys = ep->keys;
    if (ep->qkv) {
        const QkvStoreEpi& src = *ep->qkv;
        if (src.hd != BN || a.epi != 0) return false;
        a.epi = 3;
        a.qkv.q_tiles = src.q_heads;
        a.qkv.n_kv = src.kv_heads;
        a.qkv.q_norm = src.q_norm;
        a.qkv.k_norm = src.k_norm;
        a.qkv.rope = src.rope;
        a.qkv.max_pos = src.max_pos;
        a.qkv.q_out = reinterpret_cast<__nv_bfloat16*>(src.q_out);
        a.qkv.Kc = reinterpret_cast<__nv_bfloat16*>(src.Kc);
        a.qkv.Vc = reinterpret_cast<__nv_bfloat16*>(src.Vc);
        a.qkv.kv = src.kv;
        a.qkv.page_table = src.page_table;
        a.qkv.row_seq = src.row_seq;
        a.qkv.row_pos = src.row_pos;
        a.qkv.layer_tiles = src.q_heads + 2 * src.kv_heads;
        a.qkv.layer_stride = src.layer_stride;
        a.qkv.norm_stride = src.norm_stride;
        if (src.layers < 1 || N != src.layers * (src.q_heads + 2 * src.kv_heads) * BN) return false;
        if (src.layers > 1 && src.q_heads != 0) return false;  // stacked layers: context K/V only
    }
    if (a.ss_out && a.epi != 0) return false;
    if (a.epi == 2 && !a.keys) return false;
    // Passes of more than 256 rows (no row sums of squares there: the fused norm that reads
    // them serves blocks of at most 32 rows).  Measured at 512 rows on Qwen3-8B shapes: when the
    // 128 x 256 tiles fill at least one wave of the GPU the persistent kernel with whole tiles
    // wins (its epilogue overlaps the next tile's main loop); under one wave it wins only for long
    // K, with stream-K balancing (W_c, down); short-K GEMMs under one wave (QKV, O, context K/V)
    // keep the per-tile kernel below.
    if (!norm_a && a.epi != 3 && M > 256) {
        const int p_mtiles = (M + 255) / 256, p_ntiles = (N + BN - 1) / BN, KB = (K + BK - 1) / BK;
        const long long T = (long long)p_mtiles * p_ntiles;
        const int G = std::max(1, sm_count() / p_mtiles) * p_mtiles;
        if (T >= G || KB >= 128)
            return gemm_tc_persistent(L, A, lda, a_rows, W, M, N, K, C, ldc, accumulate, a.epi, a.out, a.ldo, a.keys,
                                      /*stream_k=*/T < G);
    }
    const int m_tiles = (M + MT - 1) / MT;
    if (norm_a) {
        if (MT == 16) return launch_tc<16, 4, true>(L, mw, mx, a, m_tiles);
        return launch_tc<32, 3, true>(L, mw, mx, a, m_tiles);
    }
    switch (MT) {
        case 16: return launch_tc<16, 6, false>(L, mw, mx, a, m_tiles);
        case 32: return launch_tc<32, 5, false>(L, mw, mx, a, m_tiles);
        case 64: return launch_tc<64, 4, false>(L, mw, mx, a, m_tiles);
        case 128: return launch_tc<128, 4, false>(L, mw, mx, a, m_tiles);
        default: return launch_tc<256, 4, false>(L, mw, mx, a, m_tiles);
    }
}

}  // namespace dfl
