// Internal launcher interface between the C-ABI layer (api.cu) and the kernel
// translation units.  Each launcher enqueues its kernel(s) on ctx.stream and
// bumps ctx.launches once per kernel launched.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace dfl {

struct Launch {
    cudaStream_t stream;
    long long* launches;        // incremented once per kernel launch (may be null)
    float* ws = nullptr;        // stream-K partial tiles (null: whole tiles only)
    size_t ws_bytes = 0;
    int* counters = nullptr;    // stream-K tile counters, zero between launches
    int n_counters = 0;
    uint32_t* err = nullptr;    // device error word
    bool* failed = nullptr;     // host flag: a launch could not be prepared
    bool pdl = false;           // launch with programmatic stream serialization
    void bump(int n = 1) const {
        if (launches) *launches += n;
    }
    void fail() const {
        if (failed) *failed = true;
    }
};

// Launch `kernel` on L.stream with cudaLaunchKernelEx: programmatic dependent
// launch when L.pdl is set, and a (1, 1, cluster_z) thread-block cluster when
// cluster_z > 1.  Counts the launch; a launch error sets the host flag.
template <typename... KArgs, typename... Args>
void launch_k(const Launch& L, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, int cluster_z,
              Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = L.stream;
    cudaLaunchAttribute attr[2];
    int n = 0;
    if (L.pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (cluster_z > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = 1;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = (unsigned)cluster_z;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    if (cudaLaunchKernelEx(&cfg, kernel, args...) != cudaSuccess) L.fail();
    L.bump();
}

// ---- GEMM: C[M, N] (fp32, row stride ldc) = or += A[M, K] (T, stride lda) . W[N, K]^T.
// K, lda and the W row length are multiples of 8; A and W are 16-byte aligned.
// bf16 runs on the tensor cores (gemm_tc.cu), fp32 on CUDA-core FMA (gemm.cu).
template <typename T>
void gemm(const Launch& L, const T* A, int lda, const T* W, int M, int N, int K, float* C, int ldc, bool accumulate);

// Options of the tcgen05 GEMM beyond C (=|+=) A.W^T:
//  - x_f32 set: the A operand is the fp32 matrix x [M, K] (row stride ldx) normalised on
//    the fly, A = bf16(x * rstd[m] * norm_w[k]) with rstd[m] = 1/sqrt(sum_t ss_in[t*ss_ld+m]/K + eps)
//    (blocks of at most 32 rows); the A/lda arguments are ignored;
//  - epi 1: SwiGLU; W holds gate and up rows in alternating groups of eight (rows 16g..16g+7
//    are gate rows 8g..8g+7, rows 16g+8..16g+15 the matching up rows); out[m * ldo + f] =
//    bf16(silu(gate_f) * up_f); C is unused;
//  - ss_out set (epi 0): ss_out[tile * ss_ld + m] = sum over the tile's 128 columns of C[m][n]^2
//    after the update, for the next fused norm;
//  - epi 2: row argmax: keys[m] = max_n argmax_key(C[m][n], n) by atomicMax (keys start at zero; C is
//    still written when non-null).
// q/k/v epilogue of the tcgen05 GEMM (head_dim 128): the GEMM's N columns are q_heads
// query heads, then kv_heads key heads, then kv_heads value heads (q_heads may be 0).
struct QkvStoreEpi {
    int q_heads, kv_heads, hd;
    const float* q_norm;   // [hd] or nullptr
    const float* k_norm;   // [hd] or nullptr
    const float2* rope;    // [max_pos][hd/2]
    int max_pos;
    void* q_out;           // bf16 [M, q_heads * hd]
    void* Kc;              // cache layer base (bf16)
    void* Vc;
    KVLayout kv;
    const int* page_table;
    const int* row_seq;    // [M]; < 0 = skip
    const int* row_pos;
    // Several layers in one GEMM (the drafter's context K/V): N = layers * (q_heads +
    // 2 * kv_heads) * hd; the tiles of layer l store into Kc / Vc + l * layer_stride
    // elements with k_norm + l * norm_stride.
    int layers = 1;
    long long layer_stride = 0;
    int norm_stride = 0;
};

struct GemmEpi {
    const float* x_f32 = nullptr;
    int ldx = 0;
    const float* norm_w = nullptr;
    const float* ss_in = nullptr;
    int ss_tiles = 0;
    int ss_ld = 0;
    float eps = 0.f;
    int epi = 0;
    void* out = nullptr;
    int ldo = 0;
    float* ss_out = nullptr;
    unsigned long long* keys = nullptr;  // epi 2: per-row argmax keys (zeroed by the caller)
    const QkvStoreEpi* qkv = nullptr;    // epi 3: norm + RoPE + store of q/k/v heads (C unused)
};

// tcgen05 GEMM for bf16; false when it could not be launched (tensor map encode
// failed or an unsupported option combination).  Passes of more than 256 rows without
// the fused norm or the q/k/v epilogue may run on the persistent kernel (gemm_persistent.cu),
// which writes no row sums of squares (ss_out) and uses L.ws / L.counters for stream-K
// partial tiles.
bool gemm_tc(const Launch& L, const bf16* A, int lda, int a_rows, const bf16* W, int M, int N, int K, float* C,
             int ldc, bool accumulate, const GemmEpi* ep = nullptr);
// The persistent kernel itself: epi 0 (C =|+=), 1 (SwiGLU to out), 2 (row argmax keys, C
// written when non-null); stream_k false: whole 128 x 256 tiles only.
bool gemm_tc_persistent(const Launch& L, const bf16* A, int lda, int a_rows, const bf16* W, int M, int N, int K,
                        float* C, int ldc, bool accumulate, int epi, void* out, int ldo, unsigned long long* keys,
                        bool stream_k);

// ---- row kernels
// Rows of the embedding table; with ss_out, also the per-128-column-tile sums of
// squares of each row (ss_out[tile * ss_ld + row]) for the fused norm of the next GEMM.
// d must be at most 64 * 128.
template <typename T>
void embed_rows(const Launch& L, const int* tokens, const T* embed, int vocab, int d, int rows, float* x,
                uint32_t* err, float* ss_out = nullptr, int ss_ld = 0);
template <typename T>
void rmsnorm_rows(const Launch& L, const float* x, int ldx, const float* w, int rows, int d, float eps, T* out,
                  int ldo);
// Per-row RMSNorm of rows gathered by index (row_idx[i] -> x row), used for the
// last prompt row of each sequence before the head.
template <typename T>
void rmsnorm_gather(const Launch& L, const float* x, int ldx, const int* row_idx, const float* w, int rows, int d,
                    float eps, T* out, int ldo);

struct QKVStore {
    const float* qkv;     // [rows, ld] fp32 GEMM output
    int ld;
    int q_off, k_off, v_off;  // column offsets; q_off < 0: no query heads in this pass
    int H, Hkv, hd;
    const int* row_seq;   // [rows]; < 0 = padding row (skipped)
    const int* row_pos;   // [rows]
    const float* q_norm;  // [hd] or nullptr
    const float* k_norm;  // [hd] or nullptr
    float eps;
    const float2* rope;   // [max_pos][hd/2] (cos, sin)
    int max_pos;
    void* q_out;          // T [rows, H*hd] or nullptr
    void* Kc;             // cache layer base (T)
    void* Vc;
    KVLayout kv;
    const int* page_table;
    int rows;
    uint32_t* err;
};
template <typename T>
void qk_norm_rope_store(const Launch& L, const QKVStore& p);

template <typename T>
void silu_mul(const Launch& L, const float* gu, int F, int rows, T* out);

// Copy fp32 residual rows into a bf16/fp32 staging buffer at column offset col
// (context-layer capture): stage[r * ld_stage + col + c] = x[r * d + c].
template <typename T>
void capture_rows(const Launch& L, const float* x, int d, int rows, T* stage, int ld_stage, int col);

// Token ids from argmax keys: out[r] = index(keys[r]); with block > 0 (draft rows), only rows
// r with r % block != 0 are written, to out[(r / block) * (block - 1) + r % block - 1].
void keys_to_ids(const Launch& L, const unsigned long long* keys, int rows, int block, int* out);

// Row argmax over logits [rows, V] (row stride ld); lowest index wins on ties.
void argmax_rows(const Launch& L, const float* logits, long long ld, int rows, int V, int* out);

// ---- attention
struct AttnParams {
    const void* q;        // T [rows, H*hd]
    const void* Kc;       // cache layer base
    const void* Vc;
    KVLayout kv;
    const int* page_table;
    const int* row_seq;   // [rows]
    const int* row_pos;   // [rows]
    const int* seq_len;   // non-causal: keys [0, seq_len[s] + extra); causal: nullptr, keys [0, pos]
    int extra;
    int rows;
    int group_rows;       // rows per query group (all from one sequence)
    int seq_div = 0;      // > 0: rows are sequence-major with seq_div rows each, so the sequence of
                          // row r is r / seq_div (row_seq < 0 still marks an inactive sequence)
    int H, Hkv, hd;
    int max_keys;         // host upper bound on keys seen by any row
    const int* stable_len = nullptr;  // with seq_div: keys [0, stable_len[s]) of sequence s were written
                                      // before the launch (earlier passes or joined streams), so their
                                      // tiles may load before the dependency wait; nullptr: none
    void* out;            // T [rows, H*hd]
    float* ws;            // split workspace (fp32)
    size_t ws_bytes;
};
template <typename T>
void attention(const Launch& L, const AttnParams& p);
// bf16 path of attention(): tensor cores (mma.sync), cluster-merged key splits; query groups
// of at most 64 vectors (group_rows * H / H_kv <= 64).
void attention_mma(const Launch& L, const AttnParams& p, int sms);
// Causal prefill attention on tcgen05 (attention_prefill.cu): head_dim 128, query groups of
// exactly 128 vectors (group_rows * H / H_kv == 128); false when it cannot be launched.
bool attention_prefill_tc(const Launch& L, const AttnParams& p);

// ---- temperature sampling (sampling.cu)
// Sampling settings in device memory (captured passes read them at replay):
// temperatures of the draft and verify laws, top-p (1: off) and top-k (0: off).
struct SampleParams {
    float t_draft, t_verify, top_p;
    int32_t top_k;
};
// A filtered law softmax(l / T) of one logit row: m = max l, s = sum of exp((l - m) / T)
// over the kept tokens; token z is kept when (rank key of l[z], z) ranks at or above
// (tkey, tid): key > tkey, or key == tkey and z <= tid.
struct LawStat {
    float m, s;
    uint32_t tkey;
    int32_t tid;
};
// Whether a vocabulary of V tokens fits the law clusters (each CTA stages its chunk).
bool sampling_vocab_ok(int V);
// Draft rows s*B + j (j = 1..B-1) of dlogits [batch*B, V]: dstat[row] = the filtered law
// q_j, drafts[s*(B-1) + j-1] = inverse-CDF draw of q_j with u_draft[s*(B-1) + j-1].
void draft_sample(const Launch& L, const float* dlogits, int V, int batch, int B, const SampleParams* prm,
                  const float* u_draft, LawStat* dstat, int* drafts);
// Target laws tstat[row] of every verify row, then per sequence: acceptance of the
// proposals with min(1, p/q) against u_verify[s*B + j], the residual or bonus draw with
// u_verify[s*B + B-1], and the round's bookkeeping (as accept()).
void verify_sample(const Launch& L, const float* logits, const float* dlogits, int V, int batch, int B,
                   const SampleParams* prm, const int* proposal, const float* u_verify, LawStat* tstat,
                   const LawStat* dstat, int* n, int* anchor, int* accepted, int* bonus, int* ctx_row_seq,
                   int* ctx_row_pos);

// ---- KV page table updates during the rounds (kernels.cu): table[idx[i]] = page[i], i < n
struct PageUpdates {
    int n;
    int idx[64];
    int page[64];
};
void set_pages(const Launch& L, int* table, const PageUpdates& u);

// ---- round bookkeeping
// Block rows of a draft (proposal == nullptr) or verify pass: token of row
// s*B+j is anchor[s] (j == 0), the mask id (draft) or proposal[s*(B-1)+j-1]
// (verify); position n[s]+j.
void block_rows(const Launch& L, int batch, int B, const int* n, const int* anchor, const int* proposal,
                int mask, int vocab, int max_pos, int* tokens, int* row_seq, int* row_pos, uint32_t* err);

// Greedy acceptance ([review] §4.1): a_s, bonus_s, n_s += a_s + 1, anchor_s = bonus_s,
// and the context rows to append next (row s*B+j for j <= a_s at position n_old+j).
void accept(const Launch& L, int batch, int B, const int* proposal, const int* posterior, int* n, int* anchor,
            int* accepted, int* bonus, int* ctx_row_seq, int* ctx_row_pos);

// Text returned by dflash_last_error(NULL) (calls that have no session).
__attribute__((visibility("hidden"))) void set_global_error(const char* msg);

// Gather int32 from a device array by index (used to read the last prompt row's argmax).
void fill_prefill_rows(const Launch& L, int seq, int start_pos, int rows, int* row_seq, int* row_pos);

}  // namespace dfl
