// Persistent stream-K tensor-core GEMM for passes of more than 256 token rows
// (the concurrency-32 round's 512-row verify and draft passes, 2048-row prefill
// chunks):
//
//     C[M, N] (fp32, row stride ldc)  =|+=  A[M, K] (bf16) . W[N, K]^T (bf16)
//
// As in the per-tile GEMM (gemm_tc.cu) the weights are the MMA's A operand
// (128 weight rows per tile, one output feature per TMEM lane) and the tokens
// its B operand, here always 256 per tile, so one tcgen05.mma is 128 x 256 x 16.
// A tile is one (weight tile, token tile) pair; tiles are numbered with the
// token tiles fastest so the token tiles of one weight tile run together and
// share its L2 copy.
//
// One CTA per SM walks a fixed list of work segments (no atomics decide the
// schedule, so a launch always computes the same sums in the same order):
//  - whole tiles, dealt round-robin (tile c, c + G, ...): every tile when the
//    caller asks for whole tiles only, else all full waves but the last;
//  - stream-K: the remaining weight tiles' K blocks as one flat range cut into
//    equal pieces, one per group of m_tiles CTAs (one CTA per token tile, so the
//    group reads each weight k-block at about the same time and shares its L2
//    copy); a piece may end inside a tile and the next group continues it.
//    Each piece of a split tile parks its fp32 partial sums in a workspace slot
//    and counts itself in the tile's counter; the CTA that brings the count to
//    the number of pieces adds the pieces in piece order (deterministic) and
//    applies the epilogue, then resets the counter for the next launch.  That
//    CTA is almost always at its last segment (a tile's first piece ends a
//    group's range), where the stage memory is idle: the other pieces come in
//    by bulk copies and its own piece straight from TMEM.
//
// Warp roles (192 threads): warp 0 issues TMA loads, warp 1 allocates TMEM and
// issues tcgen05.mma, warps 2-5 drain accumulators (warp w reads TMEM lanes
// 32 (w % 4) .. + 31).  TMEM holds two 256-column accumulators, so the epilogue
// of one segment overlaps the main loop of the next.  A four-stage ring of
// shared-memory stages (one 16 KB weight tile + one 32 KB token tile, 128-byte
// swizzled by TMA) is guarded by full/empty mbarriers, the accumulators by
// acc_full/acc_empty.
//
// Epilogues: fp32 C (= or +=), SwiGLU (gate and up rows alternate in groups of
// eight, so a feature's two values sit eight lanes apart and meet by one warp
// shuffle) written as bf16, and the head's row argmax (keys by atomicMax; C
// written as well when given).
//
// Every mbarrier wait is bounded; a wait that runs out sets ERR_TIMEOUT in the
// error word and the CTA stops issuing work, releases its TMEM and returns.
#include <string.h>

#include <algorithm>

#include "launch.h"
#include "tcgen05.cuh"

namespace dfl {

namespace {

using namespace tc;

constexpr int PBN = 128;                   // weight rows per tile (UMMA M)
constexpr int PMT = 256;                   // tokens per tile (UMMA N)
constexpr int PBK = 64;                    // K per stage (one 128-byte swizzle row of bf16)
constexpr int PSTAGES = 4;
constexpr int PTHREADS = 192;
constexpr int W_BYTES = PBN * PBK * 2;     // 16 KB
constexpr int X_BYTES = PMT * PBK * 2;     // 32 KB
constexpr int STAGE_BYTES = W_BYTES + X_BYTES;
constexpr int BAR_OFF = PSTAGES * STAGE_BYTES;
constexpr int NBAR = 2 * PSTAGES + 6;      // full, empty, acc_full[2], acc_empty[2], drain, fixup
constexpr int KEYS_OFF = BAR_OFF + NBAR * 8 + 16;          // wkey [4][PMT] u64 (epi 2); SwiGLU staging (epi 1)
constexpr int FLAG_OFF = KEYS_OFF + 4 * PMT * 8;
constexpr int SMEM_TOTAL = FLAG_OFF + 16 + 1024;           // + alignment slack
constexpr uint32_t TMEM_COLS = 2 * PMT;

struct PArgs {
    float* C;
    int ldc, M, N, K;
    int accumulate;
    int epi;                 // 0: C =|+=; 1: SwiGLU -> out (bf16); 2: row argmax keys (+ C if non-null)
    void* out;
    int ldo;
    unsigned long long* keys;
    uint32_t* err;
    int m_tiles, KB;
    int dp_tiles;            // tiles [0, dp_tiles) are whole-tile work, dealt round-robin
    long long sk_units;      // stream-K weight tiles * KB units, shared by groups of m_tiles CTAs
    int maxseg;              // workspace slots per stream-K tile
    float* ws;               // [sk_tiles * maxseg][PMT][PBN] partial tiles
    int* counters;           // [sk_tiles], zero between launches
};

// One piece of work: tile `tile`, K blocks [kb0, kb1); sk < 0 for a whole tile,
// else its stream-K tile index, piece number and piece count.
struct Seg {
    int tile, kb0, kb1, sk, piece, npieces;
};

// The work list of one CTA, identical for the three warp roles.  Stream-K work is
// shared by groups of m_tiles CTAs: the CTAs of a group take the same K range of the
// same weight tiles, one token tile each, so they read each weight k-block at about
// the same time and share its L2 copy.
struct Walker {
    const PArgs* a;
    int grp, NG, mt;     // group index, number of groups, this CTA's token tile
    int dp_next;         // next whole tile
    int G;
    long long u, u1;     // stream-K units [u, u1) of (weight tile, k block)

    __device__ Walker(const PArgs* a_, int cta, int G_) : a(a_), dp_next(cta), G(G_) {
        NG = G / a->m_tiles;
        grp = cta / a->m_tiles;
        mt = cta % a->m_tiles;
        u = grp < NG ? start(grp) : 0;
        u1 = grp < NG ? start(grp + 1) : 0;
    }
    __device__ long long start(int g) const { return (long long)g * a->sk_units / NG; }
    __device__ int owner(long long unit) const {  // the group whose range holds `unit`
        int g = (int)(unit * NG / (a->sk_units > 0 ? a->sk_units : 1));
        if (g > NG - 1) g = NG - 1;
        while (g + 1 < NG && start(g + 1) <= unit) ++g;
        while (g > 0 && start(g) > unit) --g;
        return g;
    }
    // whether a segment follows the one last returned
    __device__ bool more() const {
        Walker w2 = *this;
        Seg t;
        return w2.next(t);
    }
    __device__ bool next(Seg& s) {
        if (dp_next < a->dp_tiles) {
            s.tile = dp_next;
            s.kb0 = 0;
            s.kb1 = a->KB;
            s.sk = -1;
            s.piece = 0;
            s.npieces = 1;
            dp_next += G;
            return true;
        }
        if (u >= u1) return false;
        const int wt = (int)(u / a->KB);  // stream-K weight tile
        s.tile = a->dp_tiles + wt * a->m_tiles + mt;
        s.kb0 = (int)(u % a->KB);
        const long long left = u1 - u;
        s.kb1 = (int)((long long)s.kb0 + left < a->KB ? s.kb0 + left : a->KB);
        const long long first = (long long)wt * a->KB;
        const int o0 = owner(first), o1 = owner(first + a->KB - 1);
        s.npieces = o1 - o0 + 1;
        s.piece = grp - o0;
        s.sk = s.npieces > 1 ? wt * a->m_tiles + mt : -1;
        u += s.kb1 - s.kb0;
        return true;
    }
};

__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__global__ void __launch_bounds__(PTHREADS, 1)
    tc_gemm_persistent_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                              PArgs a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + BAR_OFF);
    uint64_t* empty = full + PSTAGES;
    uint64_t* acc_full = empty + PSTAGES;
    uint64_t* acc_empty = acc_full + 2;
    uint64_t* drain = acc_empty + 2;  // the MMA thread's last tcgen05 operations completed
    uint64_t* fixbar = drain + 1;     // bulk loads of other pieces' partial sums (fix-up)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + BAR_OFF + NBAR * 8);
    unsigned long long* wkey = reinterpret_cast<unsigned long long*>(smem + KEYS_OFF);
    int* last_flag = reinterpret_cast<int*>(smem + FLAG_OFF);
    int* abort_flag = last_flag + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x;

    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmW);
        prefetch_tmap(&tmX);
        for (int s = 0; s < PSTAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], 128);
        }
        mbar_init(drain, 1);
        mbar_init(fixbar, 1);
        mbar_fence_init();
        *abort_flag = 0;
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *tmem_slot;

    pdl_trigger();

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pw = policy_evict_first(), px = policy_evict_last();
            Walker wk(&a, blockIdx.x, G);
            Seg sg;
            long long it = 0;
            bool ok = true;
            bool have = wk.next(sg);
            // the first stages' weight tiles do not depend on the previous kernel: they load
            // before the wait for it, the token tiles after
            const int pre = have ? min(PSTAGES, sg.kb1 - sg.kb0) : 0;
            {
                const int nt = have ? sg.tile / a.m_tiles : 0;
                for (int i = 0; i < pre; ++i) {
                    mbar_arrive_expect_tx(&full[i], STAGE_BYTES);
                    tma_load_2d(smem + i * STAGE_BYTES, &tmW, &full[i], (sg.kb0 + i) * PBK, nt * PBN, pw);
                }
            }
            pdl_wait();
            if (have) {
                const int mt = sg.tile % a.m_tiles;
                for (int i = 0; i < pre; ++i)
                    tma_load_2d(smem + i * STAGE_BYTES + W_BYTES, &tmX, &full[i], (sg.kb0 + i) * PBK, mt * PMT, px);
                it = pre;
            }
            int kb_first = have ? sg.kb0 + pre : 0;
            while (ok && have) {
                const int nt = sg.tile / a.m_tiles, mt = sg.tile % a.m_tiles;
                for (int kb = kb_first; kb < sg.kb1; ++kb, ++it) {
                    const int s = (int)(it % PSTAGES);
                    if (it >= PSTAGES && !mbar_wait(&empty[s], (uint32_t)(((it / PSTAGES) + 1) & 1), a.err)) {
                        ok = false;
                        break;
                    }
                    uint8_t* st = smem + s * STAGE_BYTES;
                    mbar_arrive_expect_tx(&full[s], STAGE_BYTES);
                    tma_load_2d(st, &tmW, &full[s], kb * PBK, nt * PBN, pw);
                    tma_load_2d(st + W_BYTES, &tmX, &full[s], kb * PBK, mt * PMT, px);
                }
                have = wk.next(sg);
                kb_first = have ? sg.kb0 : 0;
            }
            // every load issued has landed before the CTA can exit (the MMA thread waits for
            // them in normal operation; after a timed-out wait they may still be in flight)
            for (long long i = it > PSTAGES ? it - PSTAGES : 0; i < it; ++i)
                mbar_wait(&full[i % PSTAGES], (uint32_t)((i / PSTAGES) & 1), a.err);
        }
        pdl_wait();
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16(PBN, PMT);
            Walker wk(&a, blockIdx.x, G);
            Seg sg;
            long long it = 0;
            int li = 0;
            bool ok = true;
            while (ok && wk.next(sg)) {
                const int ab = li & 1;
                if (li >= 2 && !mbar_wait(&acc_empty[ab], (uint32_t)(((li >> 1) + 1) & 1), a.err)) break;
                fence_after();
                const uint32_t d = tmem + (uint32_t)(ab * PMT);
                for (int kb = sg.kb0; kb < sg.kb1; ++kb, ++it) {
                    const int s = (int)(it % PSTAGES);
                    if (!mbar_wait(&full[s], (uint32_t)((it / PSTAGES) & 1), a.err)) {
                        ok = false;
                        break;
                    }
                    fence_after();
                    const uint32_t sw = smem_u32(smem + s * STAGE_BYTES);
                    const uint32_t sx = sw + W_BYTES;
#pragma unroll
                    for (int kk = 0; kk < PBK / 16; ++kk)
                        umma_bf16(d, sw128_desc(sw + kk * 32), sw128_desc(sx + kk * 32), idesc,
                                  (kb > sg.kb0 || kk > 0) ? 1u : 0u);
                    umma_commit(&empty[s]);
                }
                umma_commit(&acc_full[ab]);
                ++li;
            }
            // the MMAs issued above have finished before TMEM is released
            umma_commit(drain);
            mbar_wait(drain, 0, a.err);
        }
        pdl_wait();
    } else {
        // ------------------------------------------------------------ epilogue warps
        pdl_wait();  // C (accumulate) and the keys were written by earlier kernels
        const int q = warp & 3;
        const int row = 32 * q + lane;  // weight row within the tile = TMEM lane
        const int e = threadIdx.x - 64;
        const int epi = a.epi;
        const bool accum = a.accumulate != 0;
        const size_t ldc = (size_t)a.ldc;
        Walker wk(&a, blockIdx.x, G);
        Seg sg;
        int li = 0;
        int fix_phase = 0;
        while (wk.next(sg)) {
            const int ab = li & 1;
            // the four warps leave together when a wait runs out (they meet at named barriers)
            if (lane == 0 && !mbar_wait(&acc_full[ab], (uint32_t)((li >> 1) & 1), a.err)) atomicOr(abort_flag, 1);
            epi_sync();
            if (*(volatile int*)abort_flag) break;
            fence_after();
            const int nt = sg.tile / a.m_tiles, mt = sg.tile % a.m_tiles;
            const int n0 = nt * PBN, m0 = mt * PMT;
            const int n = n0 + row;
            const bool n_ok = n < a.N;
            const int m_left = a.M - m0;
            const uint32_t tbase = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(ab * PMT);

            // How this segment's final values are formed:
            //   0  a whole tile: the accumulator in TMEM;
            //   1  the last piece of a split tile, and this CTA's last segment: the stage memory is
            //      free, so the other pieces' partial sums come in by bulk copies, this piece's own
            //      from TMEM (no later MMA reuses it);
            //   2  the last piece of a split tile with more work after it: every piece from the
            //      workspace by register loads;
            //  -1  a piece that is not the last to arrive: it only parks its partial sums.
            int mode = 0;
            const float* parts = nullptr;  // piece 0's slot (the others follow at PMT * PBN strides)
            if (sg.sk >= 0) {
                const bool last_seg = !wk.more();
                // park this piece's partial sums: slot [token][row], coalesced over the warp
                float* slot = a.ws + ((size_t)sg.sk * a.maxseg + sg.piece) * (size_t)(PMT * PBN);
#pragma unroll 1
                for (int c = 0; c < PMT; c += 16) {
                    float v[16];
                    tmem_ld16(tbase + c, v);
#pragma unroll
                    for (int j = 0; j < 16; ++j) __stcg(slot + (size_t)(c + j) * PBN + row, v[j]);
                }
                fence_before();
                mbar_arrive(&acc_empty[ab]);
                __threadfence();
                epi_sync();
                if (e == 0) {
                    const int old = atomicAdd(a.counters + sg.sk, 1);
                    *last_flag = (old == sg.npieces - 1) ? 1 : 0;
                }
                epi_sync();
                if (*last_flag) {
                    __threadfence();
                    parts = a.ws + (size_t)sg.sk * a.maxseg * (size_t)(PMT * PBN);
                    mode = last_seg ? 1 : 2;
                } else {
                    mode = -1;
                }
            }
            if (mode >= 0) {
                constexpr int CH = 64;  // tokens per fix-up chunk: 32 KB of partial sums per piece
                // mode 1: as many chunks of the other pieces as fit the 192 KB of stage memory are
                // requested at once (all four for a tile split in two)
                const int others = sg.npieces - 1;
                const int batch = mode == 1 ? min(PMT / CH, (PSTAGES * STAGE_BYTES / (CH * PBN * 4)) / max(others, 1)) : 1;
#pragma unroll 1
                for (int c0 = 0; c0 < PMT; c0 += CH) {
                    const int bi = (c0 / CH) % batch;  // position of this chunk in its batch
                    if (mode == 1 && bi == 0) {
                        const int nb = min(batch, (PMT - c0) / CH);
                        if (e == 0) {
                            fence_proxy_async();  // the previous batch's reads are done (barrier below)
                            mbar_arrive_expect_tx(fixbar, (uint32_t)(nb * others * CH * PBN * 4));
                            for (int b2 = 0; b2 < nb; ++b2)
                                for (int p = 0, k = 0; p < sg.npieces; ++p) {
                                    if (p == sg.piece) continue;
                                    bulk_load(smem + (size_t)(b2 * others + k) * (CH * PBN * 4),
                                              parts + (size_t)p * (PMT * PBN) + (size_t)(c0 + b2 * CH) * PBN,
                                              (uint32_t)(CH * PBN * 4), fixbar);
                                    ++k;
                                }
                        }
                        if (!mbar_wait(fixbar, (uint32_t)(fix_phase & 1), a.err)) atomicOr(abort_flag, 1);
                        ++fix_phase;
                    }
#pragma unroll 1
                    for (int c = c0; c < c0 + CH; c += 32) {
                        // 32 tokens per step: the residual (accumulate) loads are issued first so that
                        // their round trip overlaps the reads of the sums
                        float old[32];
                        float* dst = a.C + (size_t)(m0 + c) * ldc + n;
                        if (epi == 0 && accum) {
#pragma unroll
                            for (int j = 0; j < 32; ++j) old[j] = (n_ok && c + j < m_left) ? dst[j * ldc] : 0.f;
                        }
                        float v[32];
                        if (mode == 0) {
                            uint32_t r0[16], r1[16];
                            tmem_ld16_issue(tbase + c, r0);
                            tmem_ld16_issue(tbase + c + 16, r1);
                            tmem_ld_wait(r0);
                            tmem_ld_wait(r1);
#pragma unroll
                            for (int j = 0; j < 16; ++j) {
                                v[j] = __uint_as_float(r0[j]);
                                v[16 + j] = __uint_as_float(r1[j]);
                            }
                        } else if (mode == 1) {
                            // pieces in piece order: the sum does not depend on which piece finishes
                            const float* fx = reinterpret_cast<const float*>(smem) +
                                              (size_t)bi * others * (CH * PBN) + (size_t)(c - c0) * PBN + row;
                            for (int p = 0, k = 0; p < sg.npieces; ++p) {
                                float t[32];
                                if (p == sg.piece) {
                                    uint32_t r0[16], r1[16];
                                    tmem_ld16_issue(tbase + c, r0);
                                    tmem_ld16_issue(tbase + c + 16, r1);
                                    tmem_ld_wait(r0);
                                    tmem_ld_wait(r1);
#pragma unroll
                                    for (int j = 0; j < 16; ++j) {
                                        t[j] = __uint_as_float(r0[j]);
                                        t[16 + j] = __uint_as_float(r1[j]);
                                    }
                                } else {
#pragma unroll
                                    for (int j = 0; j < 32; ++j) t[j] = fx[(size_t)k * (CH * PBN) + (size_t)j * PBN];
                                    ++k;
                                }
#pragma unroll
                                for (int j = 0; j < 32; ++j) v[j] = p == 0 ? t[j] : v[j] + t[j];
                            }
                        } else {
                            for (int p0 = 0; p0 < sg.npieces; p0 += 2) {
                                float t[2][32];
#pragma unroll
                                for (int pp = 0; pp < 2; ++pp)
                                    if (p0 + pp < sg.npieces) {
                                        const float* src = parts + (size_t)(p0 + pp) * (PMT * PBN) + (size_t)c * PBN + row;
#pragma unroll
                                        for (int j = 0; j < 32; ++j) t[pp][j] = __ldcg(src + (size_t)j * PBN);
                                    }
#pragma unroll
                                for (int pp = 0; pp < 2; ++pp)
                                    if (p0 + pp < sg.npieces) {
#pragma unroll
                                        for (int j = 0; j < 32; ++j) v[j] = (p0 + pp == 0) ? t[pp][j] : v[j] + t[pp][j];
                                    }
                            }
                        }
                        if (epi == 0) {
                            if (n_ok) {
                                if (accum) {
#pragma unroll
                                    for (int j = 0; j < 32; ++j)
                                        if (c + j < m_left) dst[j * ldc] = old[j] + v[j];
                                } else {
#pragma unroll
                                    for (int j = 0; j < 32; ++j)
                                        if (c + j < m_left) dst[j * ldc] = v[j];
                                }
                            }
                        } else if (epi == 1) {
                            // gate rows 16g .. 16g+7, up rows 16g+8 .. 16g+15: lane and lane ^ 8.  The
                            // warp's 16 features x 32 tokens go through a 1 KB shared buffer [token][feature]
                            // so that each lane then writes whole 16-byte runs of a token's features
                            // (two stores per lane instead of 32 narrow ones).
                            // The gate lane and its up lane split the 32 tokens: the gate lane evaluates
                            // tokens 0..15, the up lane tokens 16..31, after swapping the halves they need.
                            __nv_bfloat16* sb = reinterpret_cast<__nv_bfloat16*>(wkey) + q * (32 * 16);
                            const bool gate = (row & 8) == 0;
                            const int fl = ((lane >> 4) << 3) | (lane & 7);  // the pair's feature, 0..15
                            const int t0 = gate ? 0 : 16;
#pragma unroll
                            for (int j = 0; j < 16; ++j) {
                                const float x = __shfl_xor_sync(0xffffffffu, gate ? v[16 + j] : v[j], 8);
                                const float g = gate ? v[j] : x;        // gate value of token t0 + j
                                const float u = gate ? x : v[16 + j];   // up value of token t0 + j
                                sb[(t0 + j) * 16 + fl] = __float2bfloat16_rn(__fdividef(g, 1.f + __expf(-g)) * u);
                            }
                            __syncwarp();
                            const int F = a.N >> 1;
#pragma unroll
                            for (int i = 0; i < 2; ++i) {
                                const int id = lane + 32 * i, tok = id >> 1, hf = id & 1;
                                const int f0 = 64 * nt + 16 * q + 8 * hf;
                                const uint4 val = *reinterpret_cast<const uint4*>(sb + tok * 16 + hf * 8);
                                if (f0 < F && c + tok < m_left)
                                    *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.out) +
                                                              (size_t)(m0 + c + tok) * a.ldo + f0) = val;
                            }
                            __syncwarp();  // the buffer is rewritten by the next step
                        } else {
#pragma unroll
                            for (int half = 0; half < 2; ++half) {
                                unsigned long long k[16];
#pragma unroll
                                for (int j = 0; j < 16; ++j) {
                                    const int jj = 16 * half + j;
                                    const bool live = n_ok && c + jj < m_left;
                                    k[j] = live ? argmax_key(v[jj], (uint32_t)n) : 0ull;
                                    if (a.C && live) a.C[(size_t)(m0 + c + jj) * ldc + n] = v[jj];
                                }
                                const unsigned long long best = transpose_reduce16(
                                    k, lane, [](unsigned long long x, unsigned long long y) { return x > y ? x : y; });
                                if (!(lane & 1)) wkey[q * PMT + c + 16 * half + (lane >> 1)] = best;
                            }
                        }
                    }
                    if (mode == 1 && (bi == batch - 1 || c0 + CH == PMT))
                        epi_sync();  // every read of this batch is done before the next copies
                }
                if (mode == 0) {
                    fence_before();
                    mbar_arrive(&acc_empty[ab]);
                }
                if (epi == 2) {
                    epi_sync();
                    for (int j = e; j < PMT; j += 128) {
                        unsigned long long best = wkey[j];
#pragma unroll
                        for (int w2 = 1; w2 < 4; ++w2) best = wkey[w2 * PMT + j] > best ? wkey[w2 * PMT + j] : best;
                        if (j < m_left) atomicMax(a.keys + m0 + j, best);
                    }
                    epi_sync();  // wkey is rewritten by the next tile
                }
                if (parts && e == 0) a.counters[sg.sk] = 0;  // ready for the next launch
            }
            ++li;
        }
    }

    fence_before();
    __syncthreads();
    if (warp == 1) {
        fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

}  // namespace

// Whole tiles for every full wave but the last; stream-K over the rest.  Returns
// false when the launch cannot be prepared (nothing is launched).
bool gemm_tc_persistent(const Launch& L, const bf16* A, int lda, int a_rows, const bf16* W, int M, int N, int K,
                        float* C, int ldc, bool accumulate, int epi, void* out, int ldo, unsigned long long* keys,
                        bool stream_k) {
    if (M <= 0 || N <= 0 || K <= 0) return true;
    static bool attr = false;
    if (!attr) {
        if (cudaFuncSetAttribute(tc_gemm_persistent_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SMEM_TOTAL) != cudaSuccess)
            return false;
        attr = true;
    }
    CUtensorMap mw, mx;
    if (!tc::make_map(&mw, W, N, K, K, PBN)) return false;
    if (!tc::make_map(&mx, A, a_rows, K, lda, PMT)) return false;
    PArgs a;
    memset(&a, 0, sizeof a);
    a.C = C;
    a.ldc = ldc;
    a.M = M;
    a.N = N;
    a.K = K;
    a.accumulate = accumulate ? 1 : 0;
    a.epi = epi;
    a.out = out;
    a.ldo = ldo;
    a.keys = keys;
    a.err = L.err;
    a.m_tiles = (M + PMT - 1) / PMT;
    a.KB = (K + PBK - 1) / PBK;
    const int n_tiles = (N + PBN - 1) / PBN;
    const long long T = (long long)n_tiles * a.m_tiles;
    // the grid is a whole number of CTA groups (one CTA per token tile in a group)
    int G = std::max(1, tc::sm_count() / a.m_tiles) * a.m_tiles;
    // whole tiles for all full waves but the last one; the last wave and the remainder are
    // balanced by stream-K (a remainder of at least 7/8 of a wave runs as whole tiles too)
    long long waves = T / G, rem = T % G;
    long long dp_waves = (rem == 0 || rem * 8 >= 7LL * G) ? waves + (rem ? 1 : 0) : (waves > 0 ? waves - 1 : 0);
    long long dp = std::min<long long>(dp_waves * G, T);        // a multiple of m_tiles (or T)
    long long sk_ntiles = n_tiles - dp / a.m_tiles;
    long long units = sk_ntiles * a.KB;
    int NG = G / a.m_tiles;
    // with stream-K work only, fewer groups when the pieces would fall under 8 K blocks (each
    // piece costs a 128 KB partial-tile round trip), but never fewer than one per weight tile
    if (dp == 0) {
        NG = (int)std::min<long long>(NG, std::max<long long>(sk_ntiles, (units + 7) / 8));
        G = NG * a.m_tiles;
    }
    int maxseg = 1;
    if (sk_ntiles > 0) {
        // pieces per stream-K tile (owner groups of its first and last K block)
        auto start = [&](long long g) { return g * units / NG; };
        auto owner = [&](long long u) {
            long long g = u * NG / units;
            if (g > NG - 1) g = NG - 1;
            while (g + 1 < NG && start(g + 1) <= u) ++g;
            while (g > 0 && start(g) > u) --g;
            return g;
        };
        for (long long t = 0; t < sk_ntiles; ++t)
            maxseg = (int)std::max<long long>(maxseg, owner(t * a.KB + a.KB - 1) - owner(t * a.KB) + 1);
    }
    const long long sk_tiles = sk_ntiles * a.m_tiles;
    const size_t ws_need = (size_t)sk_tiles * maxseg * PMT * PBN * sizeof(float);
    // (the fix-up holds the other pieces' 32 KB chunks in the stage memory: at most 6 of them)
    if (sk_tiles > 0 && (maxseg > 7 || ws_need > L.ws_bytes || sk_tiles > L.n_counters || !L.ws || !L.counters)) {
        // no room for the partial tiles: whole tiles only
        dp = T;
        units = 0;
        maxseg = 1;
    }
    if (!stream_k) {
        dp = T;
        units = 0;
        maxseg = 1;
    }
    a.dp_tiles = (int)dp;
    a.sk_units = units;
    a.maxseg = maxseg;
    a.ws = L.ws;
    a.counters = L.counters;
    if (dp == T && T < G) G = (int)T;
    launch_k(L, tc_gemm_persistent_kernel, dim3(G), dim3(PTHREADS), (size_t)SMEM_TOTAL, 1, mw, mx, a);
    return true;
}

}  // namespace dfl


