// C-ABI layer: session state, weight packing, and the orchestration of
// prefill, draft_block, verify and generate on one CUDA stream.
//
// The round follows the greedy decoding-round pseudocode of "DFlash: Block
// Diffusion for Flash Speculative Decoding" (Method, Inference §4.1) and the
// verification rule of "DFlash: Why a Diffusion Drafter Can Accelerate an
// Autoregressive Model" (§4.1, Algorithm 1).  Every arithmetic step runs in
// the kernels of this library; the host only sequences launches, copies
// tokens, and keeps lengths for capacity checks.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <cmath>
#include <string>
#include <vector>

#include "dflash.h"
#include "launch.h"
#include "page_pool.h"
#include "loss.h"

using namespace dfl;

static thread_local std::string g_init_error;

namespace dfl {
void set_global_error(const char* msg) { g_init_error = msg; }
}  // namespace dfl

namespace {

constexpr int PAGE_TOKENS = 64;
constexpr int PAGE_SHIFT = 6;
constexpr int PREFILL_CHUNK = 2048;
constexpr size_t ATTN_WS_BYTES = 64ull << 20;
constexpr size_t GEMM_WS_BYTES = 96ull << 20;  // stream-K partial tiles, one workspace per stream
constexpr int GEMM_COUNTERS = 1 << 16;

enum State { ST_EMPTY = 0, ST_READY = 1, ST_DRAFTED = 2 };

struct LayerW {
    void* wqkv = nullptr;         // [(H + 2 Hkv) hd, d]: rows wq, wk, wv (library-owned copy)
    const void* wo = nullptr;     // [d, H hd] (the caller's buffer, borrowed)
    void* wgu = nullptr;          // [2F, d]: rows w_gate, w_up (library-owned copy)
    const void* wdown = nullptr;  // [d, F] (borrowed)
    float* attn_norm = nullptr;
    float* mlp_norm = nullptr;
    float* q_norm = nullptr;
    float* k_norm = nullptr;
};

}  // namespace

struct dflash_ctx {
    dflash_config cfg;
    cudaStream_t stream = nullptr;
    std::string err;
    std::vector<void*> allocs;
    long long launches = 0;
    size_t esz = 4;  // element size of the storage type

    int d, H, Hkv, hd, F, V, Lt, Ld, B, k, qd, kvd, qkv_n, max_seq;
    void* ctx_wkv = nullptr;     // bf16: [Ld * 2 kvd, d], every draft layer's wk, wv stacked (context K/V in one GEMM)
    float* ctx_knorm = nullptr;  // [Ld * hd]: the draft layers' k_norm, stacked
    int Bmax = 0;      // configured block size: every round buffer is sized for it
    int append_B = 0;  // block size of the verify whose accepted rows await the context append
    int ctx_slot[64];  // target layer -> index in ctx_layer_ids or -1

    std::vector<LayerW> tl, dl;
    // borrowed from the caller: used in place, never freed here
    const void* embed = nullptr;
    const void* head = nullptr;
    const void* fc = nullptr;
    float* final_norm = nullptr;
    float* fc_norm = nullptr;
    float* draft_norm = nullptr;

    KVLayout kv;
    void *tK = nullptr, *tV = nullptr, *dK = nullptr, *dV = nullptr;
    int* page_table = nullptr;        // [max_batch * pages_per_seq]: physical page of each (slot, logical page)
    // KV page pool (host side): physical pages [0, pool_pages) of the caches, the last one a
    // scratch page that backs every unassigned table entry (never handed out)
    int pool_pages = 0;
    PagePool pool;
    float2* rope = nullptr;

    int R = 0;  // row capacity
    float* x = nullptr;
    void* xn = nullptr;
    void* xn_ctx = nullptr;  // normalised operand of the context append (its own: it may run concurrently)
    float* qkv = nullptr;
    void* q = nullptr;
    void* att = nullptr;
    float* gu = nullptr;
    void* hmid = nullptr;
    void* stage = nullptr;
    float* fcout = nullptr;
    // temperature sampling: draft logits kept for verify, softmax row statistics,
    // uniforms and temperatures (device memory, so captured graphs stay valid)
    float* dlogits = nullptr;
    LawStat* dstat = nullptr;              // filtered draft laws of the last sampled draft
    LawStat* tstat = nullptr;              // filtered target laws of the last sampled verify
    float* u_draft = nullptr;
    float* u_verify = nullptr;
    SampleParams* prm_dev = nullptr;       // temperatures, top-p, top-k (read by the sampling kernels)
    SampleParams* prm_pinned = nullptr;    // host staging of prm_dev
    float temp_cur[2] = {-1.f, -1.f};      // temperatures last written to prm_dev
    int top_k = 0;                         // filter last written to prm_dev (0 / 1: off)
    float top_p = 1.f;
    bool draft_sampled = false;
    bool draft_logits_out = false;         // the draft pass also writes its logits to dlogits
    void* feat = nullptr;
    float* ss_x = nullptr;   // [ss_tiles][R]: per-128-column sums of squares of x rows (fused norms)
    float* ss_fc = nullptr;  // same for fcout
    int ss_tiles = 0;
    float* kvout = nullptr;
    float* logits = nullptr;
    int* tokens = nullptr;
    int* row_seq = nullptr;
    int* row_pos = nullptr;
    int* ctx_row_seq = nullptr;
    int* ctx_row_pos = nullptr;
    int* n = nullptr;
    int* anchor = nullptr;
    int* proposal = nullptr;
    int* posterior = nullptr;
    int* argbuf = nullptr;
    unsigned long long* keys = nullptr;  // head argmax keys [max_batch * B]
    int* accepted = nullptr;
    int* bonus = nullptr;
    int* drafts = nullptr;
    uint32_t* errw = nullptr;
    float* attn_ws = nullptr;
    float* gemm_ws = nullptr;
    int* gemm_counters = nullptr;
    float* gemm_ws_side = nullptr;     // the same for GEMMs on side_stream (they may run concurrently)
    int* gemm_counters_side = nullptr;
    bool launch_failed = false;
    float* keep_prefill = nullptr;
    float* keep_draft = nullptr;
    float* keep_verify = nullptr;
    float* keep_hidden = nullptr;

    int batch = 0;
    int state = ST_EMPTY;
    bool pending_append = false;
    std::vector<int> n_upper;  // host upper bound of n (exact after a synchronising verify)

    dflash_stats stats;
    cudaEvent_t ev[4];
    bool events = false;

    // kernel-class profile (DFLASH_FLAG_PROFILE)
    struct ProfRec {
        int kind, e0, e1;
        long long launches;
        double bytes, flops;
    };
    bool profiling = false;

    // CUDA graphs of the draft pass (without / with the context append) and the
    // verify pass, captured on `cap_stream` and replayed on `stream`
    struct GraphSlot {
        cudaGraphExec_t exec = nullptr;
        long long key = -1;  // (batch, block size, block size of the pending append)
        long long kernels = 0;
        int eager_runs = 0;
    };
    GraphSlot g_draft[2], g_verify, g_draft_s[2], g_verify_s;
    cudaStream_t cap_stream = nullptr;
    // The context append of a draft pass runs on `side_stream`, forked from and joined back
    // into the pass's stream: draft layer l waits only for ctx_ev[l] (its context K/V).
    cudaStream_t side_stream = nullptr;
    std::vector<cudaEvent_t> ctx_ev;  // [Ld] per-layer done, [Ld] fork point
    bool append_forked = false;
    bool graphs = true;
    std::vector<cudaEvent_t> prof_ev;
    int prof_next = 0;
    std::vector<ProfRec> prof_pending;
    dflash_profile_entry prof_acc[DFLASH_K_COUNT];

    Launch L() {
        Launch l{stream, &launches};
        const bool side = side_stream && stream == side_stream;
        l.ws = side ? gemm_ws_side : gemm_ws;
        l.ws_bytes = GEMM_WS_BYTES;
        l.counters = side ? gemm_counters_side : gemm_counters;
        l.n_counters = GEMM_COUNTERS;
        l.err = errw;
        l.failed = &launch_failed;
        l.pdl = true;
        return l;
    }

    dflash_status fail(dflash_status s, const char* fmt, ...) {
        char buf[512];
        va_list ap;
        va_start(ap, fmt);
        vsnprintf(buf, sizeof buf, fmt, ap);
        va_end(ap);
        err = buf;
        return s;
    }
};

namespace {

#define CUDA_TRY(ctx, call)                                                                   \
    do {                                                                                      \
        cudaError_t e_ = (call);                                                              \
        if (e_ != cudaSuccess)                                                                \
            return (ctx)->fail(DFLASH_E_CUDA, "%s: %s", #call, cudaGetErrorString(e_));      \
    } while (0)

void* dev_alloc(dflash_ctx* c, size_t bytes) {
    if (bytes == 0) bytes = 16;
    void* p = nullptr;
    if (c->cfg.alloc) {
        p = c->cfg.alloc(bytes, c->cfg.alloc_user);
    } else if (cudaMalloc(&p, bytes) != cudaSuccess) {
        cudaGetLastError();
        p = nullptr;
    }
    if (p) c->allocs.push_back(p);
    return p;
}

bool is_device_ptr(const void* p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

template <typename T>
T* elem(void* base, size_t offset_elems) {
    return reinterpret_cast<T*>(base) + offset_elems;
}

dflash_status validate(const dflash_config* c, std::string& why) {
    char buf[256];
    auto bad = [&](const char* m) {
        why = m;
        return DFLASH_E_INVAL;
    };
    if (c->dtype != DFLASH_DTYPE_F32 && c->dtype != DFLASH_DTYPE_BF16) return bad("dtype must be F32 or BF16");
    if (c->head_dim != 64 && c->head_dim != 128) return bad("head_dim must be 64 or 128");
    if (c->d_model <= 0 || c->d_model % 64 || c->d_model > 8192)
        return bad("d_model must be a positive multiple of 64, at most 8192");
    if (c->ffn <= 0 || c->ffn % 64) return bad("ffn must be a positive multiple of 64");
    if (c->n_heads <= 0 || c->n_kv_heads <= 0 || c->n_heads % c->n_kv_heads) return bad("n_heads % n_kv_heads != 0");
    if (c->n_heads / c->n_kv_heads > 64) return bad("more than 64 query heads per KV head");
    if (c->vocab <= 1) return bad("vocab must be > 1");
    if (c->target_layers <= 0 || c->target_layers > 64) return bad("target_layers must be in [1, 64]");
    if (c->draft_layers <= 0 || c->draft_layers > 64) return bad("draft_layers must be in [1, 64]");
    if (c->block_size < 1 || c->block_size > 32) return bad("block_size must be in [1, 32]");
    if (c->n_ctx_layers < 1 || c->n_ctx_layers > DFLASH_MAX_CTX_LAYERS) return bad("n_ctx_layers out of range");
    for (int i = 0; i < c->n_ctx_layers; ++i)
        if (c->ctx_layer_ids[i] < 0 || c->ctx_layer_ids[i] >= c->target_layers) {
            snprintf(buf, sizeof buf, "ctx_layer_ids[%d] = %d outside [0, target_layers)", i, c->ctx_layer_ids[i]);
            why = buf;
            return DFLASH_E_INVAL;
        }
    for (int i = 0; i < c->n_ctx_layers; ++i)
        for (int j = 0; j < i; ++j)
            if (c->ctx_layer_ids[i] == c->ctx_layer_ids[j]) return bad("ctx_layer_ids must be distinct");
    if (c->mask_token < 0 || c->mask_token >= c->vocab) return bad("mask_token outside [0, vocab)");
    if (c->max_batch < 1 || c->max_batch > 1024) return bad("max_batch must be in [1, 1024]");
    if (c->max_seq_len < c->block_size + 1) return bad("max_seq_len too small");
    if (c->kv_pool_tokens < 0 || c->kv_pool_tokens > (1ll << 36)) return bad("kv_pool_tokens must be in [0, 2^36]");
    if (!(c->rms_eps > 0.f) || !(c->rope_theta > 1.0)) return bad("rms_eps and rope_theta must be positive");
    if ((c->alloc == nullptr) != (c->free == nullptr)) return bad("alloc and free must both be set or both NULL");
    if ((double)c->max_batch * c->block_size * 2 * c->ffn > 2e9) return bad("batch x block x ffn too large");
    return DFLASH_OK;
}

// Copy a [rows, cols] device matrix into dst at row offset (element size esz).
dflash_status copy_rows(dflash_ctx* c, void* dst, size_t row_off, const void* src, size_t rows, size_t cols) {
    if (!src) return c->fail(DFLASH_E_INVAL, "a weight pointer is NULL");
    CUDA_TRY(c, cudaMemcpyAsync((char*)dst + row_off * cols * c->esz, src, rows * cols * c->esz,
                                cudaMemcpyDeviceToDevice, c->stream));
    return DFLASH_OK;
}

dflash_status copy_norm(dflash_ctx* c, float** dst, const float* src, size_t n, bool optional) {
    if (!src) {
        if (optional) {
            *dst = nullptr;
            return DFLASH_OK;
        }
        return c->fail(DFLASH_E_INVAL, "a norm weight pointer is NULL");
    }
    *dst = (float*)dev_alloc(c, n * 4);
    if (!*dst) return c->fail(DFLASH_E_NOMEM, "allocation of %zu bytes failed", n * 4);
    CUDA_TRY(c, cudaMemcpyAsync(*dst, src, n * 4, cudaMemcpyDeviceToDevice, c->stream));
    return DFLASH_OK;
}

// A weight used in place: non-NULL and 16-byte aligned (tensor-map and vector loads).
dflash_status borrow(dflash_ctx* c, const void** dst, const void* src, const char* what) {
    if (!src) return c->fail(DFLASH_E_INVAL, "weight %s is NULL", what);
    if ((uintptr_t)src & 15u) return c->fail(DFLASH_E_INVAL, "weight %s is not 16-byte aligned", what);
    *dst = src;
    return DFLASH_OK;
}

dflash_status pack_layer(dflash_ctx* c, const dflash_layer_weights& w, LayerW& o, bool qk_norm) {
    const size_t d = c->d, F = c->F, qd = c->qd, kvd = c->kvd;
    dflash_status s;
    if ((s = borrow(c, &o.wo, w.wo, "wo"))) return s;
    if ((s = borrow(c, &o.wdown, w.w_down, "w_down"))) return s;
    o.wqkv = dev_alloc(c, (qd + 2 * kvd) * d * c->esz);
    o.wgu = dev_alloc(c, 2 * F * d * c->esz);
    if (!o.wqkv || !o.wgu) return c->fail(DFLASH_E_NOMEM, "weight allocation failed");
    if ((s = copy_rows(c, o.wqkv, 0, w.wq, qd, d))) return s;
    if ((s = copy_rows(c, o.wqkv, qd, w.wk, kvd, d))) return s;
    if ((s = copy_rows(c, o.wqkv, qd + kvd, w.wv, kvd, d))) return s;
    if (c->cfg.dtype == DFLASH_DTYPE_BF16) {
        // SwiGLU epilogue layout: groups of 16 rows, gate rows [8g, 8g+8) then up rows [8g, 8g+8),
        // so that a 128-row GEMM tile holds both halves of 64 features, eight TMEM lanes apart
        if (!w.w_gate || !w.w_up) return c->fail(DFLASH_E_INVAL, "a weight pointer is NULL");
        const size_t blk = 8 * d * c->esz;
        CUDA_TRY(c, cudaMemcpy2DAsync(o.wgu, 2 * blk, w.w_gate, blk, blk, F / 8, cudaMemcpyDeviceToDevice, c->stream));
        CUDA_TRY(c, cudaMemcpy2DAsync((char*)o.wgu + blk, 2 * blk, w.w_up, blk, blk, F / 8, cudaMemcpyDeviceToDevice,
                                      c->stream));
    } else {
        if ((s = copy_rows(c, o.wgu, 0, w.w_gate, F, d))) return s;
        if ((s = copy_rows(c, o.wgu, F, w.w_up, F, d))) return s;
    }
    if ((s = copy_norm(c, &o.attn_norm, w.attn_norm, d, false))) return s;
    if ((s = copy_norm(c, &o.mlp_norm, w.mlp_norm, d, false))) return s;
    if (qk_norm) {
        if ((s = copy_norm(c, &o.q_norm, w.q_norm, c->hd, false))) return s;
        if ((s = copy_norm(c, &o.k_norm, w.k_norm, c->hd, false))) return s;
    }
    return DFLASH_OK;
}

// Device error word -> status (synchronises).
dflash_status check_device(dflash_ctx* c) {
    uint32_t e = 0;
    CUDA_TRY(c, cudaMemcpyAsync(&e, c->errw, 4, cudaMemcpyDeviceToHost, c->stream));
    CUDA_TRY(c, cudaStreamSynchronize(c->stream));
    if (e) {
        CUDA_TRY(c, cudaMemsetAsync(c->errw, 0, 4, c->stream));
        if (e & ERR_TIMEOUT) {
            // a GEMM that stopped early may have left stream-K tile counters raised
            CUDA_TRY(c, cudaMemsetAsync(c->gemm_counters, 0, (size_t)GEMM_COUNTERS * 4, c->stream));
            CUDA_TRY(c, cudaMemsetAsync(c->gemm_counters_side, 0, (size_t)GEMM_COUNTERS * 4, c->stream));
            return c->fail(DFLASH_E_TIMEOUT, "a bounded device-side wait ran out (code %u)", e);
        }
        return c->fail(DFLASH_E_DEVICE_CHECK, "device-side check failed (code %u%s%s)", e,
                       (e & ERR_TOKEN_RANGE) ? ": token id outside [0, vocab)" : "",
                       (e & ERR_POSITION_RANGE) ? ": position beyond max_seq_len" : "");
    }
    return DFLASH_OK;
}

// Fold recorded event pairs into the per-class profile (synchronises).
dflash_status prof_drain(dflash_ctx* c) {
    if (c->prof_pending.empty()) return DFLASH_OK;
    CUDA_TRY(c, cudaEventSynchronize(c->prof_ev[c->prof_pending.back().e1]));
    for (const auto& r : c->prof_pending) {
        float ms = 0.f;
        CUDA_TRY(c, cudaEventElapsedTime(&ms, c->prof_ev[r.e0], c->prof_ev[r.e1]));
        dflash_profile_entry& a = c->prof_acc[r.kind];
        a.launches += r.launches;
        a.ms += ms;
        a.bytes += r.bytes;
        a.flops += r.flops;
    }
    c->prof_pending.clear();
    c->prof_next = 0;
    return DFLASH_OK;
}

// Run f (which enqueues kernels of one class); with profiling on, bracket it
// with events and remember its algorithmic bytes and flops.
template <class F>
void timed(dflash_ctx* c, int kind, double bytes, double flops, F&& f) {
    if (!c->profiling) {
        f();
        return;
    }
    if (c->prof_next + 2 > (int)c->prof_ev.size()) prof_drain(c);
    const int e0 = c->prof_next++, e1 = c->prof_next++;
    const long long l0 = c->launches;
    cudaEventRecord(c->prof_ev[e0], c->stream);
    f();
    cudaEventRecord(c->prof_ev[e1], c->stream);
    c->prof_pending.push_back({kind, e0, e1, c->launches - l0, bytes, flops});
}

double gemm_bytes(const dflash_ctx* c, double M, double N, double K, bool acc) {
    return N * K * c->esz + M * K * c->esz + M * N * 4.0 * (acc ? 2.0 : 1.0);
}

int attn_group_rows(int rows_per_seq, int g) {
    int best = 1;
    for (int r = 1; r <= rows_per_seq; ++r)
        if (rows_per_seq % r == 0 && r * g <= 64) best = r;
    return best;
}

dflash_status launch_check(dflash_ctx* c);

// ------------------------------------------------------------ model passes
template <typename T>
struct Pass {
    dflash_ctx* c;

    KVLayout kvl() const { return c->kv; }

    static constexpr bool is_bf16 = sizeof(T) == 2;

    // C (or the SwiGLU output `out`) = rms_norm(x, norm_w) . W^T for `rows` rows of the
    // fp32 matrix x (row stride K).  bf16 blocks of <= 32 rows normalise inside the GEMM
    // (sums of squares from ss_in, left there by the kernel that wrote x); otherwise an
    // RMSNorm kernel writes the bf16/fp32 operand first.
    // `fusable` false: the row sums of squares in ss_in may be stale (the rows were last written
    // by a pass of more than 256 rows, whose persistent GEMM writes none), so normalise first.
    void normed_gemm(int kind, int rows, const float* x, const float* norm_w, const float* ss_in, const T* W, int N,
                     int K, float* C, int ldc, T* out, int ldo, unsigned long long* keys = nullptr,
                     const QkvStoreEpi* qkv = nullptr, void* xbuf = nullptr, bool fusable = true) {
        void* xn = xbuf ? xbuf : c->xn;
        Launch L = c->L();
        const double R = rows, es = c->esz;
        const double bytes = (double)N * K * es + R * K * 4 + (out ? R * ldo * es : R * N * 4.0);
        const bool fused = is_bf16 && rows <= 32 && fusable;
        if (!fused)
            timed(c, DFLASH_K_NORM, R * K * (4 + es), 0, [&] {
                rmsnorm_rows<T>(L, x, K, norm_w, rows, K, c->cfg.rms_eps, (T*)xn, K);
            });
        timed(c, kind, bytes, 2 * R * N * (double)K, [&] {
            if constexpr (sizeof(T) == 2) {
                GemmEpi e;
                if (fused) {
                    e.x_f32 = x;
                    e.ldx = K;
                    e.norm_w = norm_w;
                    e.ss_in = ss_in;
                    e.ss_tiles = c->ss_tiles;
                    e.ss_ld = c->R;
                    e.eps = c->cfg.rms_eps;
                }
                if (out) {
                    e.epi = 1;
                    e.out = out;
                    e.ldo = ldo;
                }
                if (keys) {
                    e.epi = 2;
                    e.keys = keys;
                }
                e.qkv = qkv;
                if (!gemm_tc(L, (const bf16*)xn, K, rows, (const bf16*)W, rows, N, K, C, ldc, false, &e)) L.fail();
            } else {
                gemm<T>(L, (const T*)xn, K, W, rows, N, K, C, ldc, false);
            }
        });
    }

    // q/k norm, RoPE and the cache store run in the projection GEMM's epilogue for
    // bf16 blocks of <= 32 rows with head_dim 128 (one head per 128-row weight tile).
    bool qkv_in_epilogue(int rows) const { return is_bf16 && rows <= 32 && c->hd == 128; }

    QkvStoreEpi qkv_epi(int q_heads, const float* q_norm, const float* k_norm, void* Kc, void* Vc,
                        const int* row_seq, const int* row_pos) const {
        QkvStoreEpi e;
        e.q_heads = q_heads;
        e.kv_heads = c->Hkv;
        e.hd = c->hd;
        e.q_norm = q_norm;
        e.k_norm = k_norm;
        e.rope = reinterpret_cast<const float2*>(c->rope);
        e.max_pos = c->max_seq;
        e.q_out = c->q;
        e.Kc = Kc;
        e.Vc = Vc;
        e.kv = c->kv;
        e.page_table = c->page_table;
        e.row_seq = row_seq;
        e.row_pos = row_pos;
        return e;
    }

    // x += A . W^T (residual update); bf16 also leaves the sums of squares of the
    // updated rows in ss_x for the next fused norm.
    void residual_gemm(int kind, int rows, const T* A, int K, const T* W, int lda) {
        Launch L = c->L();
        const double R = rows, d = c->d;
        timed(c, kind, gemm_bytes(c, R, d, K, true), 2 * R * d * (double)K, [&] {
            if constexpr (sizeof(T) == 2) {
                GemmEpi e;
                e.ss_out = c->ss_x;
                e.ss_ld = c->R;
                if (!gemm_tc(L, (const bf16*)A, lda, rows, (const bf16*)W, rows, c->d, K, c->x, c->d, true, &e)) L.fail();
            } else {
                gemm<T>(L, A, lda, W, rows, c->d, K, c->x, c->d, true);
            }
        });
    }

    // Decoder layers over `rows` rows whose metadata is (row_seq, row_pos).
    // target: causal attention over the target cache, capture of context layers
    // into stage; draft: bidirectional attention over [context ; block].
    void layers(bool target, int rows, const int* row_seq, const int* row_pos, int group_rows, int max_keys,
                bool capture, double keys_total, int rows_per_seq = 0, const int* stable_len = nullptr) {
        Launch L = c->L();
        const int nl = target ? c->Lt : c->Ld;
        const double R = rows, d = c->d, es = c->esz;
        for (int l = 0; l < nl; ++l) {
            const LayerW& w = target ? c->tl[l] : c->dl[l];
            void* Kc = elem<T>(target ? c->tK : c->dK, (size_t)l * c->kv.layer_stride);
            void* Vc = elem<T>(target ? c->tV : c->dV, (size_t)l * c->kv.layer_stride);
            const bool fuse_qkv = qkv_in_epilogue(rows);
            const QkvStoreEpi qe = qkv_epi(c->H, w.q_norm, w.k_norm, Kc, Vc, row_seq, row_pos);
            normed_gemm(DFLASH_K_GEMM_QKV, rows, c->x, w.attn_norm, c->ss_x, (const T*)w.wqkv, c->qkv_n, c->d,
                        c->qkv, c->qkv_n, nullptr, 0, nullptr, fuse_qkv ? &qe : nullptr);
            QKVStore st;
            st.qkv = c->qkv;
            st.ld = c->qkv_n;
            st.q_off = 0;
            st.k_off = c->qd;
            st.v_off = c->qd + c->kvd;
            st.H = c->H;
            st.Hkv = c->Hkv;
            st.hd = c->hd;
            st.row_seq = row_seq;
            st.row_pos = row_pos;
            st.q_norm = w.q_norm;
            st.k_norm = w.k_norm;
            st.eps = c->cfg.rms_eps;
            st.rope = c->rope;
            st.max_pos = c->max_seq;
            st.q_out = c->q;
            st.Kc = Kc;
            st.Vc = Vc;
            st.kv = c->kv;
            st.page_table = c->page_table;
            st.rows = rows;
            st.err = c->errw;
            if (!fuse_qkv)
                timed(c, DFLASH_K_ROPE_STORE, R * c->qkv_n * (4 + es), 0, [&] { qk_norm_rope_store<T>(L, st); });
            AttnParams ap;
            ap.q = c->q;
            ap.Kc = Kc;
            ap.Vc = Vc;
            ap.kv = c->kv;
            ap.page_table = c->page_table;
            ap.row_seq = row_seq;
            ap.row_pos = row_pos;
            ap.seq_len = target ? nullptr : c->n;
            ap.extra = target ? 0 : c->B;
            ap.rows = rows;
            ap.group_rows = group_rows;
            ap.seq_div = rows_per_seq;
            ap.H = c->H;
            ap.Hkv = c->Hkv;
            ap.hd = c->hd;
            ap.max_keys = max_keys;
            ap.stable_len = stable_len;
            ap.out = c->att;
            ap.ws = c->attn_ws;
            ap.ws_bytes = ATTN_WS_BYTES;
            // the draft's attention reads this layer's context K/V, appended on the side stream
            if (!target && c->append_forked && cudaStreamWaitEvent(c->stream, c->ctx_ev[l], 0) != cudaSuccess)
                c->launch_failed = true;
            timed(c, DFLASH_K_ATTENTION, keys_total * 2 * c->kvd * es + 2 * R * c->qd * es,
                  4.0 * R * c->H * c->hd * (keys_total / std::max(1.0, (double)c->batch)), [&] { attention<T>(L, ap); });
            residual_gemm(DFLASH_K_GEMM_O, rows, (const T*)c->att, c->qd, (const T*)w.wo, c->qd);
            if (is_bf16) {
                // gate/up GEMM with the fused norm and the SwiGLU epilogue -> hmid (bf16)
                normed_gemm(DFLASH_K_GEMM_GATE_UP, rows, c->x, w.mlp_norm, c->ss_x, (const T*)w.wgu, 2 * c->F, c->d,
                            nullptr, 0, (T*)c->hmid, c->F);
            } else {
                normed_gemm(DFLASH_K_GEMM_GATE_UP, rows, c->x, w.mlp_norm, c->ss_x, (const T*)w.wgu, 2 * c->F, c->d,
                            c->gu, 2 * c->F, nullptr, 0);
                timed(c, DFLASH_K_SWIGLU, R * c->F * (8 + es), 0,
                      [&] { silu_mul<T>(L, c->gu, c->F, rows, (T*)c->hmid); });
            }
            residual_gemm(DFLASH_K_GEMM_DOWN, rows, (const T*)c->hmid, c->F, (const T*)w.wdown, c->F);
            if (target && capture && c->ctx_slot[l] >= 0)
                timed(c, DFLASH_K_OTHER, R * d * (4 + es), 0, [&] {
                    capture_rows<T>(L, c->x, c->d, rows, (T*)c->stage, c->k * c->d, c->ctx_slot[l] * c->d);
                });
        }
    }

    // Context feature rms(W_c stage) and its K/V in every draft layer, stored
    // at (ctx_seq, ctx_pos); rows with ctx_seq < 0 are skipped.
    void append_context(int rows, const int* ctx_seq, const int* ctx_pos, cudaEvent_t* layer_done = nullptr) {
        Launch L = c->L();
        const double R = rows, d = c->d, es = c->esz;
        timed(c, DFLASH_K_GEMM_FC, gemm_bytes(c, R, d, c->k * d, false), 2 * R * d * c->k * d, [&] {
            if (is_bf16) {
                GemmEpi e;
                e.ss_out = c->ss_fc;
                e.ss_ld = c->R;
                if (!gemm_tc(L, (const bf16*)c->stage, c->k * c->d, rows, (const bf16*)c->fc, rows, c->d, c->k * c->d,
                             c->fcout, c->d, false, &e))
                    L.fail();
            } else {
                gemm<T>(L, (const T*)c->stage, c->k * c->d, (const T*)c->fc, rows, c->d, c->k * c->d, c->fcout, c->d,
                        false);
            }
        });
        if (qkv_in_epilogue(rows) && c->ctx_wkv) {
            // every draft layer's K/V of the context rows in one GEMM over the stacked weights;
            // the epilogue stores each layer's tiles (k-norm, RoPE) into that layer's cache
            QkvStoreEpi qe = qkv_epi(0, nullptr, c->ctx_knorm, c->dK, c->dV, ctx_seq, ctx_pos);
            qe.layers = c->Ld;
            qe.layer_stride = c->kv.layer_stride;
            qe.norm_stride = c->hd;
            normed_gemm(DFLASH_K_GEMM_CTX_KV, rows, c->fcout, c->fc_norm, c->ss_fc, (const T*)c->ctx_wkv,
                        c->Ld * 2 * c->kvd, c->d, c->kvout, 2 * c->kvd, nullptr, 0, nullptr, &qe, c->xn_ctx);
            if (layer_done)
                for (int l = 0; l < c->Ld; ++l)
                    if (cudaEventRecord(layer_done[l], c->stream) != cudaSuccess) c->launch_failed = true;
            return;
        }
        for (int l = 0; l < c->Ld; ++l) {
            const LayerW& w = c->dl[l];
            const T* wkv = elem<T>(w.wqkv, (size_t)c->qd * c->d);  // rows wk, wv
            // context feature rms(fcout) * fc_norm feeds every draft layer's K/V projection
            const bool fuse_kv = qkv_in_epilogue(rows);
            const QkvStoreEpi qe = qkv_epi(0, nullptr, w.k_norm, elem<T>(c->dK, (size_t)l * c->kv.layer_stride),
                                           elem<T>(c->dV, (size_t)l * c->kv.layer_stride), ctx_seq, ctx_pos);
            normed_gemm(DFLASH_K_GEMM_CTX_KV, rows, c->fcout, c->fc_norm, c->ss_fc, wkv, 2 * c->kvd, c->d, c->kvout,
                        2 * c->kvd, nullptr, 0, nullptr, fuse_kv ? &qe : nullptr, c->xn_ctx);
            QKVStore st;
            st.qkv = c->kvout;
            st.ld = 2 * c->kvd;
            st.q_off = -1;
            st.k_off = 0;
            st.v_off = c->kvd;
            st.H = c->H;
            st.Hkv = c->Hkv;
            st.hd = c->hd;
            st.row_seq = ctx_seq;
            st.row_pos = ctx_pos;
            st.q_norm = nullptr;
            st.k_norm = w.k_norm;
            st.eps = c->cfg.rms_eps;
            st.rope = c->rope;
            st.max_pos = c->max_seq;
            st.q_out = nullptr;
            st.Kc = elem<T>(c->dK, (size_t)l * c->kv.layer_stride);
            st.Vc = elem<T>(c->dV, (size_t)l * c->kv.layer_stride);
            st.kv = c->kv;
            st.page_table = c->page_table;
            st.rows = rows;
            st.err = c->errw;
            if (!fuse_kv)
                timed(c, DFLASH_K_ROPE_STORE, R * 2.0 * c->kvd * (4 + es), 0, [&] { qk_norm_rope_store<T>(L, st); });
            if (layer_done && cudaEventRecord(layer_done[l], c->stream) != cudaSuccess) c->launch_failed = true;
        }
    }

    // Final norm + shared head + row argmax over `rows` rows of x starting at row0.
    // `block` > 0: draft rows, token ids of rows s*block+j (j >= 1) go to out[s*(block-1)+j-1].
    // `logits_to` set: the fp32 logits are written there (the sampled passes), else to
    // c->logits only when kept (bf16) or always (fp32, whose argmax reads them).
    void head(int row0, int rows, const float* norm, int* out, float* keep, int block = 0, float* logits_to = nullptr,
              bool fusable = true) {
        Launch L = c->L();
        const double R = rows, V = c->V;
        float* lg = logits_to ? logits_to : c->logits;
        if (is_bf16) {
            // head GEMM with the argmax in its epilogue (logits written only when needed)
            cudaMemsetAsync(c->keys, 0, (size_t)rows * sizeof(unsigned long long), c->stream);
            normed_gemm(DFLASH_K_GEMM_HEAD, rows, c->x + (size_t)row0 * c->d, norm, c->ss_x + row0,
                        (const T*)c->head, c->V, c->d, (keep || logits_to) ? lg : nullptr, c->V, nullptr, 0, c->keys,
                        nullptr, nullptr, fusable);
            timed(c, DFLASH_K_ARGMAX, R * 8, 0, [&] { keys_to_ids(L, c->keys, rows, block, out); });
        } else {
            normed_gemm(DFLASH_K_GEMM_HEAD, rows, c->x + (size_t)row0 * c->d, norm, c->ss_x + row0,
                        (const T*)c->head, c->V, c->d, lg, c->V, nullptr, 0);
            if (block > 0) {
                timed(c, DFLASH_K_ARGMAX, R * V * 4, 0, [&] { argmax_rows(L, lg, c->V, rows, c->V, c->argbuf); });
                cudaMemcpy2DAsync(out, (size_t)(block - 1) * 4, c->argbuf + 1, (size_t)block * 4,
                                  (size_t)(block - 1) * 4, rows / block, cudaMemcpyDeviceToDevice, c->stream);
            } else {
                timed(c, DFLASH_K_ARGMAX, R * V * 4, 0, [&] { argmax_rows(L, lg, c->V, rows, c->V, out); });
            }
        }
        if (keep) cudaMemcpyAsync(keep, lg, (size_t)rows * c->V * 4, cudaMemcpyDeviceToDevice, c->stream);
    }

    dflash_status prefill(int batch, const int* lens, const int* toks, int* first) {
        Launch L = c->L();
        const int g = c->H / c->Hkv;
        size_t off = 0;
        for (int s = 0; s < batch; ++s) {
            const int P = lens[s];
            for (int r0 = 0; r0 < P; r0 += PREFILL_CHUNK) {
                const int rows = std::min(PREFILL_CHUNK, P - r0);
                CUDA_TRY(c, cudaMemcpyAsync(c->tokens, toks + off + r0, (size_t)rows * 4, cudaMemcpyHostToDevice,
                                            c->stream));
                fill_prefill_rows(L, s, r0, rows, c->row_seq, c->row_pos);
                embed_rows<T>(L, c->tokens, (const T*)c->embed, c->V, c->d, rows, c->x, c->errw, c->ss_x, c->R);
                // bf16, head_dim 128: query groups of 128 vectors for the tcgen05 prefill attention
                const int gr = (is_bf16 && c->hd == 128 && 128 % g == 0) ? 128 / g : 64 / g;
                layers(true, rows, c->row_seq, c->row_pos, gr, r0 + rows, true, (double)(r0 + rows));
                append_context(rows, c->row_seq, c->row_pos);
                if (r0 + rows == P)
                    head(rows - 1, 1, c->final_norm, c->anchor + s,
                         c->keep_prefill ? c->keep_prefill + (size_t)s * c->V : nullptr, 0, nullptr, rows <= 256);
            }
            off += P;
        }
        dflash_status ls = launch_check(c);
        if (ls != DFLASH_OK) return ls;
        std::vector<int> nh(lens, lens + batch);
        CUDA_TRY(c, cudaMemcpyAsync(c->n, nh.data(), (size_t)batch * 4, cudaMemcpyHostToDevice, c->stream));
        CUDA_TRY(c, cudaMemcpyAsync(first, c->anchor, (size_t)batch * 4, cudaMemcpyDeviceToHost, c->stream));
        return check_device(c);
    }

    // Draft pass; `sampled`: proposals drawn from softmax(draft logits / T) (T in device memory).
    void draft(bool sampled = false) {
        Launch L = c->L();
        const int b = c->batch, B = c->B, g = c->H / c->Hkv;
        c->append_forked = false;
        if (c->pending_append) {
            if (is_bf16 && !c->profiling && c->side_stream) {
                // fork: the append streams its weights while the draft layers run
                cudaStream_t main = c->stream;
                if (cudaEventRecord(c->ctx_ev[c->Ld], main) != cudaSuccess ||
                    cudaStreamWaitEvent(c->side_stream, c->ctx_ev[c->Ld], 0) != cudaSuccess)
                    c->launch_failed = true;
                c->stream = c->side_stream;
                append_context(b * c->append_B, c->ctx_row_seq, c->ctx_row_pos, c->ctx_ev.data());
                c->stream = main;
                c->append_forked = true;
            } else {
                append_context(b * c->append_B, c->ctx_row_seq, c->ctx_row_pos);
            }
            c->pending_append = false;
        }
        if (B == 1) {
            join_append();
            return;
        }
        timed(c, DFLASH_K_OTHER, (double)b * B * c->d * (4 + c->esz), 0, [&] {
            block_rows(L, b, B, c->n, c->anchor, nullptr, c->cfg.mask_token, c->V, c->max_seq, c->tokens, c->row_seq,
                       c->row_pos, c->errw);
            embed_rows<T>(L, c->tokens, (const T*)c->embed, c->V, c->d, b * B, c->x, c->errw, c->ss_x, c->R);
        });
        // attention grid sized from the session capacity, not the current length, so
        // that the pass is the same launch sequence every round (graph replay)
        double keys = 0;
        for (int s = 0; s < b; ++s) keys += c->n_upper[s] + B;
        // (the n committed context entries are complete before each layer's attention starts)
        layers(false, b * B, c->row_seq, c->row_pos, attn_group_rows(B, g), c->max_seq, false, keys, B, c->n);
        join_append();  // (already joined by the last layer's attention; kept for clarity)
        // drafts[s][j] = argmax of row s*B + 1 + j
        head(0, b * B, c->draft_norm, c->drafts, c->keep_draft, B,
             (sampled || c->draft_logits_out) ? c->dlogits : nullptr);
        if (sampled)  // drafts[s][j] = draw from q of row s*B + 1 + j (replaces the argmax)
            timed(c, DFLASH_K_SAMPLING, (double)b * (B - 1) * c->V * 4, 0, [&] {
                draft_sample(L, c->dlogits, c->V, b, B, c->prm_dev, c->u_draft, c->dstat, c->drafts);
            });
    }

    // The pass's stream waits for the whole forked append (its last event).
    void join_append() {
        if (!c->append_forked) return;
        if (cudaStreamWaitEvent(c->stream, c->ctx_ev[c->Ld - 1], 0) != cudaSuccess) c->launch_failed = true;
        c->append_forked = false;
    }

    // Verify pass; `sampled`: acceptance and emission by speculative rejection sampling.
    void verify(bool sampled = false) {
        Launch L = c->L();
        const int b = c->batch, B = c->B, g = c->H / c->Hkv;
        timed(c, DFLASH_K_OTHER, (double)b * B * c->d * (4 + c->esz), 0, [&] {
            block_rows(L, b, B, c->n, c->anchor, c->proposal, c->cfg.mask_token, c->V, c->max_seq, c->tokens,
                       c->row_seq, c->row_pos, c->errw);
            embed_rows<T>(L, c->tokens, (const T*)c->embed, c->V, c->d, b * B, c->x, c->errw, c->ss_x, c->R);
        });
        double keys = 0;
        for (int s = 0; s < b; ++s) keys += c->n_upper[s] + B;
        layers(true, b * B, c->row_seq, c->row_pos, attn_group_rows(B, g), c->max_seq, true, keys, B, c->n);
        if (c->keep_hidden)
            cudaMemcpyAsync(c->keep_hidden, c->x, (size_t)b * B * c->d * 4, cudaMemcpyDeviceToDevice, c->stream);
        head(0, b * B, c->final_norm, c->posterior, c->keep_verify, 0, sampled ? c->logits : nullptr);
        if (sampled) {
            timed(c, DFLASH_K_SAMPLING, (double)b * (B + 2) * c->V * 4, 0, [&] {
                verify_sample(L, c->logits, c->dlogits, c->V, b, B, c->prm_dev, c->proposal, c->u_verify, c->tstat,
                              c->dstat, c->n, c->anchor, c->accepted, c->bonus, c->ctx_row_seq, c->ctx_row_pos);
            });
        } else {
            timed(c, DFLASH_K_OTHER, (double)b * B * 8, 0, [&] {
                accept(L, b, B, c->proposal, c->posterior, c->n, c->anchor, c->accepted, c->bonus, c->ctx_row_seq,
                       c->ctx_row_pos);
            });
        }
        c->pending_append = true;
        c->append_B = B;
    }
};

// ---- KV page pool
// Every slot's table row returns to the scratch page and every page to the pool.
void pool_reset(dflash_ctx* c) { c->pool.reset(); }

// Back positions [0, tokens) of `slot` with pages; false when the pool runs out.
bool pool_ensure(dflash_ctx* c, int slot, long long tokens) { return c->pool.ensure(slot, tokens, PAGE_TOKENS); }

// The device page table follows the host mirror, in stream order: after a reset the whole table
// (a pageable copy, which may wait for the stream: prefill, init and the training forward only);
// between rounds the few new entries, written by a kernel that carries them in its parameters,
// so that the rounds stay asynchronous.
dflash_status pool_upload(dflash_ctx* c) {
    const PagePool& P = c->pool;
    if (P.full_dirty()) {
        CUDA_TRY(c, cudaMemcpyAsync(c->page_table, P.table().data(), P.table().size() * 4, cudaMemcpyHostToDevice,
                                    c->stream));
        c->pool.uploaded();
        return DFLASH_OK;
    }
    Launch L = c->L();
    const std::vector<int>& pend = P.pending();
    for (size_t i = 0; i < pend.size(); i += 64) {
        PageUpdates u;
        u.n = (int)std::min<size_t>(64, pend.size() - i);
        for (int j = 0; j < u.n; ++j) {
            u.idx[j] = pend[i + j];
            u.page[j] = P.table()[pend[i + j]];
        }
        set_pages(L, c->page_table, u);
    }
    c->pool.uploaded();
    return launch_check(c);
}

dflash_status pool_full(dflash_ctx* c, int slot, long long tokens) {
    return c->fail(DFLASH_E_CAPACITY, "KV page pool exhausted: sequence %d needs %lld tokens (%d pages of %d in use)",
                   slot, tokens, c->pool.in_use(), c->pool.capacity());
}

dflash_status capacity_check(dflash_ctx* c) {
    for (int s = 0; s < c->batch; ++s) {
        if (c->n_upper[s] + c->B > c->cfg.max_seq_len) {
            // refresh from the device before refusing
            std::vector<int> nh(c->batch);
            CUDA_TRY(c, cudaMemcpyAsync(nh.data(), c->n, (size_t)c->batch * 4, cudaMemcpyDeviceToHost, c->stream));
            CUDA_TRY(c, cudaStreamSynchronize(c->stream));
            c->n_upper = nh;
            if (c->n_upper[s] + c->B > c->cfg.max_seq_len)
                return c->fail(DFLASH_E_CAPACITY, "sequence %d: length %d + block %d exceeds max_seq_len %d", s,
                               c->n_upper[s], c->B, c->cfg.max_seq_len);
        }
    }
    // pages for every position the round may write (the block at n .. n+B-1)
    for (int s = 0; s < c->batch; ++s)
        if (!pool_ensure(c, s, (long long)c->n_upper[s] + c->B)) {
            std::vector<int> nh(c->batch);  // the bound may be loose: refresh it from the device first
            CUDA_TRY(c, cudaMemcpyAsync(nh.data(), c->n, (size_t)c->batch * 4, cudaMemcpyDeviceToHost, c->stream));
            CUDA_TRY(c, cudaStreamSynchronize(c->stream));
            c->n_upper = nh;
            if (!pool_ensure(c, s, (long long)c->n_upper[s] + c->B)) return pool_full(c, s, (long long)c->n_upper[s] + c->B);
        }
    return pool_upload(c);
}

dflash_status launch_check(dflash_ctx* c) {
    if (c->launch_failed) {
        c->launch_failed = false;
        return c->fail(DFLASH_E_CUDA, "a tensor-core GEMM could not be prepared (TMA descriptor encode failed)");
    }
    CUDA_TRY(c, cudaGetLastError());
    return DFLASH_OK;
}

void reset_graph(dflash_ctx::GraphSlot& g) {
    if (g.exec) cudaGraphExecDestroy(g.exec);
    g = dflash_ctx::GraphSlot();
}

// Run one pass: eagerly the first time (and whenever profiling), then as a
// captured CUDA graph.  Every launch of a pass reads the round's variable state
// (lengths, anchors, proposals) from device memory and uses grids fixed by the
// session's capacity, so a captured pass replays the same work as an eager one.
template <class F>
dflash_status run_pass(dflash_ctx* c, dflash_ctx::GraphSlot& g, F&& pass) {
    if (!c->graphs || c->profiling) {
        pass();
        return launch_check(c);
    }
    const long long key = ((long long)c->batch << 16) | (c->B << 8) | (c->pending_append ? c->append_B : 0);
    if (g.exec && g.key == key) {
        CUDA_TRY(c, cudaGraphLaunch(g.exec, c->stream));
        c->launches += g.kernels;
        // host-side effects of the pass
        return DFLASH_OK;
    }
    if (g.key != key) {
        reset_graph(g);
        g.key = key;
    }
    if (g.eager_runs < 1) {
        ++g.eager_runs;
        pass();
        return launch_check(c);
    }
    // capture on the library's own stream, ordered after the caller's stream
    cudaStream_t user = c->stream;
    CUDA_TRY(c, cudaEventRecord(c->ev[3], user));
    CUDA_TRY(c, cudaStreamWaitEvent(c->cap_stream, c->ev[3], 0));
    CUDA_TRY(c, cudaStreamBeginCapture(c->cap_stream, cudaStreamCaptureModeThreadLocal));
    c->stream = c->cap_stream;
    const long long l0 = c->launches;
    pass();
    c->stream = user;
    cudaGraph_t graph = nullptr;
    cudaError_t e = cudaStreamEndCapture(c->cap_stream, &graph);
    if (e != cudaSuccess || !graph) return c->fail(DFLASH_E_CUDA, "graph capture failed: %s", cudaGetErrorString(e));
    dflash_status ls = launch_check(c);
    if (ls != DFLASH_OK) {
        cudaGraphDestroy(graph);
        return ls;
    }
    e = cudaGraphInstantiate(&g.exec, graph, 0);
    cudaGraphDestroy(graph);
    if (e != cudaSuccess) {
        g.exec = nullptr;
        return c->fail(DFLASH_E_CUDA, "graph instantiation failed: %s", cudaGetErrorString(e));
    }
    g.kernels = c->launches - l0;
    CUDA_TRY(c, cudaGraphLaunch(g.exec, c->stream));
    return DFLASH_OK;
}

dflash_status do_draft(dflash_ctx* c, bool sampled = false) {
    const int with_append = c->pending_append ? 1 : 0;
    dflash_status s = run_pass(c, sampled ? c->g_draft_s[with_append] : c->g_draft[with_append], [&] {
        if (c->cfg.dtype == DFLASH_DTYPE_BF16) Pass<bf16>{c}.draft(sampled);
        else Pass<float>{c}.draft(sampled);
    });
    c->pending_append = false;
    return s;
}

dflash_status do_verify(dflash_ctx* c, bool sampled = false) {
    dflash_status s = run_pass(c, sampled ? c->g_verify_s : c->g_verify, [&] {
        if (c->cfg.dtype == DFLASH_DTYPE_BF16) Pass<bf16>{c}.verify(sampled);
        else Pass<float>{c}.verify(sampled);
    });
    if (s != DFLASH_OK) return s;
    c->pending_append = true;
    c->append_B = c->B;
    for (int i = 0; i < c->batch; ++i) c->n_upper[i] += c->B;
    return DFLASH_OK;
}

// Stage user tokens [b, B-1] into ctx->proposal.
dflash_status load_proposal(dflash_ctx* c, const int32_t* toks) {
    const size_t n = (size_t)c->batch * (c->B - 1);
    if (n == 0) return DFLASH_OK;
    if (toks == c->drafts) {
        CUDA_TRY(c, cudaMemcpyAsync(c->proposal, toks, n * 4, cudaMemcpyDeviceToDevice, c->stream));
    } else if (is_device_ptr(toks)) {
        CUDA_TRY(c, cudaMemcpyAsync(c->proposal, toks, n * 4, cudaMemcpyDeviceToDevice, c->stream));
    } else {
        for (size_t i = 0; i < n; ++i)
            if (toks[i] < 0 || toks[i] >= c->V)
                return c->fail(DFLASH_E_INVAL, "draft token %zu = %d outside [0, %d)", i, toks[i], c->V);
        CUDA_TRY(c, cudaMemcpyAsync(c->proposal, toks, n * 4, cudaMemcpyHostToDevice, c->stream));
    }
    return DFLASH_OK;
}

// Stage n caller uniforms (host or device) into dst; host values must lie in [0, 1).
dflash_status load_uniforms(dflash_ctx* c, float* dst, const float* u, size_t n) {
    if (n == 0) return DFLASH_OK;
    if (is_device_ptr(u)) {
        CUDA_TRY(c, cudaMemcpyAsync(dst, u, n * 4, cudaMemcpyDeviceToDevice, c->stream));
    } else {
        for (size_t i = 0; i < n; ++i)
            if (!(u[i] >= 0.f && u[i] < 1.f)) return c->fail(DFLASH_E_INVAL, "uniform %zu = %g outside [0, 1)", i, u[i]);
        CUDA_TRY(c, cudaMemcpyAsync(dst, u, n * 4, cudaMemcpyHostToDevice, c->stream));
    }
    return DFLASH_OK;
}

// The temperature reaches the kernels through device memory (captured passes stay valid);
// it is copied only when it changes, from pinned memory, after the stream has drained any
// copy of the previous value.
dflash_status set_temperature(dflash_ctx* c, int which, float t) {
    if (!(t > 0.f) || !std::isfinite(t)) return c->fail(DFLASH_E_INVAL, "temperature %g is not a positive finite number", t);
    if (c->temp_cur[which] == t) return DFLASH_OK;
    CUDA_TRY(c, cudaStreamSynchronize(c->stream));
    float* host = which == 0 ? &c->prm_pinned->t_draft : &c->prm_pinned->t_verify;
    float* dev = which == 0 ? &c->prm_dev->t_draft : &c->prm_dev->t_verify;
    *host = t;
    CUDA_TRY(c, cudaMemcpyAsync(dev, host, 4, cudaMemcpyHostToDevice, c->stream));
    c->temp_cur[which] = t;
    return DFLASH_OK;
}

dflash_status store_out(dflash_ctx* c, void* dst, const void* src, size_t bytes, bool* host) {
    *host = false;
    if (bytes == 0 || dst == src) return DFLASH_OK;
    if (is_device_ptr(dst)) {
        CUDA_TRY(c, cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, c->stream));
    } else {
        CUDA_TRY(c, cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToHost, c->stream));
        *host = true;
    }
    return DFLASH_OK;
}

}  // namespace

// ===================================================================== C ABI
extern "C" {

dflash_status dflash_init(const dflash_config* cfg, const dflash_weights* w, void* cuda_stream, dflash_ctx** out) {
    if (!out) return DFLASH_E_INVAL;
    *out = nullptr;
    if (!cfg || !w || !w->target || !w->draft) {
        g_init_error = "cfg, weights and layer arrays must be non-NULL";
        return DFLASH_E_INVAL;
    }
    std::string why;
    if (validate(cfg, why) != DFLASH_OK) {
        g_init_error = why;
        return DFLASH_E_INVAL;
    }
    dflash_ctx* c = new dflash_ctx();
    c->cfg = *cfg;
    c->stream = (cudaStream_t)cuda_stream;
    memset(&c->stats, 0, sizeof c->stats);
    c->esz = cfg->dtype == DFLASH_DTYPE_BF16 ? 2 : 4;
    c->d = cfg->d_model;
    c->H = cfg->n_heads;
    c->Hkv = cfg->n_kv_heads;
    c->hd = cfg->head_dim;
    c->F = cfg->ffn;
    c->V = cfg->vocab;
    c->Lt = cfg->target_layers;
    c->Ld = cfg->draft_layers;
    c->B = cfg->block_size;
    c->Bmax = cfg->block_size;
    c->k = cfg->n_ctx_layers;
    c->qd = c->H * c->hd;
    c->kvd = c->Hkv * c->hd;
    c->qkv_n = c->qd + 2 * c->kvd;
    c->max_seq = (cfg->max_seq_len + PAGE_TOKENS - 1) / PAGE_TOKENS * PAGE_TOKENS;
    for (int l = 0; l < 64; ++l) c->ctx_slot[l] = -1;
    for (int i = 0; i < c->k; ++i) c->ctx_slot[cfg->ctx_layer_ids[i]] = i;

    auto bail = [&](dflash_status s) {
        g_init_error = c->err;
        dflash_destroy(c);
        return s;
    };
#define ALLOC(ptr, bytes)                                                                   \
    do {                                                                                    \
        (ptr) = (decltype(ptr))dev_alloc(c, (bytes));                                       \
        if (!(ptr)) {                                                                       \
            c->fail(DFLASH_E_NOMEM, "device allocation of %zu bytes failed", (size_t)(bytes)); \
            return bail(DFLASH_E_NOMEM);                                                    \
        }                                                                                   \
    } while (0)

    const size_t d = c->d, V = c->V, esz = c->esz;
    // weights: embedding, head, W_c, wo and w_down are used in place; wq/wk/wv and
    // w_gate/w_up are packed into library-owned matrices
    dflash_status s;
    if ((s = borrow(c, &c->embed, w->embed, "embed"))) return bail(s);
    if ((s = borrow(c, &c->head, w->head, "head"))) return bail(s);
    if ((s = borrow(c, &c->fc, w->fc, "fc"))) return bail(s);
    if ((s = copy_norm(c, &c->final_norm, w->final_norm, d, false))) return bail(s);
    if ((s = copy_norm(c, &c->fc_norm, w->fc_norm, d, false))) return bail(s);
    if ((s = copy_norm(c, &c->draft_norm, w->draft_norm, d, false))) return bail(s);
    c->tl.resize(c->Lt);
    c->dl.resize(c->Ld);
    for (int l = 0; l < c->Lt; ++l)
        if ((s = pack_layer(c, w->target[l], c->tl[l], cfg->target_qk_norm != 0))) return bail(s);
    for (int l = 0; l < c->Ld; ++l)
        if ((s = pack_layer(c, w->draft[l], c->dl[l], true))) return bail(s);
    if (cfg->dtype == DFLASH_DTYPE_BF16 && c->hd == 128) {
        // the context K/V of every draft layer comes from the same feature: one stacked GEMM
        c->ctx_wkv = dev_alloc(c, (size_t)c->Ld * 2 * c->kvd * d * c->esz);
        c->ctx_knorm = (float*)dev_alloc(c, (size_t)c->Ld * c->hd * 4);
        if (!c->ctx_wkv || !c->ctx_knorm) return bail(c->fail(DFLASH_E_NOMEM, "weight allocation failed"));
        for (int l = 0; l < c->Ld; ++l) {
            if ((s = copy_rows(c, c->ctx_wkv, (size_t)l * 2 * c->kvd, w->draft[l].wk, c->kvd, d))) return bail(s);
            if ((s = copy_rows(c, c->ctx_wkv, (size_t)l * 2 * c->kvd + c->kvd, w->draft[l].wv, c->kvd, d)))
                return bail(s);
            if (cudaMemcpyAsync(c->ctx_knorm + (size_t)l * c->hd, c->dl[l].k_norm, (size_t)c->hd * 4,
                                cudaMemcpyDeviceToDevice, c->stream) != cudaSuccess)
                return bail(c->fail(DFLASH_E_CUDA, "copy of the draft k-norms failed"));
        }
    }

    // caches: one pool of 64-token pages shared by the batch (plus a scratch page), assigned per
    // sequence by the host as it grows; the page table starts with every entry on the scratch page
    c->kv.page_tokens = PAGE_TOKENS;
    c->kv.page_shift = PAGE_SHIFT;
    c->kv.pages_per_seq = c->max_seq / PAGE_TOKENS;
    c->kv.n_kv_heads = c->Hkv;
    c->kv.head_dim = c->hd;
    const size_t table = (size_t)cfg->max_batch * c->kv.pages_per_seq;
    const long long pool_tokens =
        cfg->kv_pool_tokens > 0 ? cfg->kv_pool_tokens : (long long)cfg->max_batch * c->max_seq;
    c->pool_pages = (int)((pool_tokens + PAGE_TOKENS - 1) / PAGE_TOKENS) + 1;  // + the scratch page
    c->kv.layer_stride = (long long)c->pool_pages * c->Hkv * PAGE_TOKENS * c->hd;
    ALLOC(c->tK, (size_t)c->Lt * c->kv.layer_stride * esz);
    ALLOC(c->tV, (size_t)c->Lt * c->kv.layer_stride * esz);
    ALLOC(c->dK, (size_t)c->Ld * c->kv.layer_stride * esz);
    ALLOC(c->dV, (size_t)c->Ld * c->kv.layer_stride * esz);
    ALLOC(c->page_table, table * 4);
    c->pool.init(c->pool_pages, cfg->max_batch, c->kv.pages_per_seq);
    if (pool_upload(c) != DFLASH_OK || cudaStreamSynchronize(c->stream) != cudaSuccess) {
        c->fail(DFLASH_E_CUDA, "page table upload failed");
        return bail(DFLASH_E_CUDA);
    }
    // RoPE table: angle pos * theta^(-2j/hd) in double, stored as fp32 (cos, sin)
    ALLOC(c->rope, (size_t)c->max_seq * (c->hd / 2) * sizeof(float2));
    {
        std::vector<float2> t((size_t)c->max_seq * (c->hd / 2));
        for (int p = 0; p < c->max_seq; ++p)
            for (int j = 0; j < c->hd / 2; ++j) {
                const double inv = pow(cfg->rope_theta, -2.0 * j / c->hd);
                const double a = (double)p * inv;
                t[(size_t)p * (c->hd / 2) + j] = make_float2((float)cos(a), (float)sin(a));
            }
        if (cudaMemcpy(c->rope, t.data(), t.size() * sizeof(float2), cudaMemcpyHostToDevice) != cudaSuccess) {
            c->fail(DFLASH_E_CUDA, "rope table upload failed");
            return bail(DFLASH_E_CUDA);
        }
    }
    // round buffers
    const int rb = cfg->max_batch * c->Bmax;
    c->R = std::max(rb, PREFILL_CHUNK);
    const size_t R = c->R;
    ALLOC(c->x, R * d * 4);
    ALLOC(c->xn, R * d * esz);
    ALLOC(c->xn_ctx, R * d * esz);
    ALLOC(c->qkv, R * c->qkv_n * 4);
    ALLOC(c->q, R * c->qd * esz);
    ALLOC(c->att, R * c->qd * esz);
    ALLOC(c->gu, R * 2 * c->F * 4);
    ALLOC(c->hmid, R * c->F * esz);
    ALLOC(c->stage, R * c->k * d * esz);
    ALLOC(c->fcout, R * d * 4);
    c->ss_tiles = (c->d + 127) / 128;
    ALLOC(c->ss_x, (size_t)c->ss_tiles * R * 4);
    ALLOC(c->ss_fc, (size_t)c->ss_tiles * R * 4);
    ALLOC(c->feat, R * d * esz);
    ALLOC(c->kvout, R * 2 * c->kvd * 4);
    ALLOC(c->logits, (size_t)rb * V * 4);
    ALLOC(c->dlogits, (size_t)rb * V * 4);
    ALLOC(c->dstat, (size_t)rb * sizeof(LawStat));
    ALLOC(c->tstat, (size_t)rb * sizeof(LawStat));
    ALLOC(c->u_draft, (size_t)rb * 4);
    ALLOC(c->u_verify, (size_t)rb * 4);
    ALLOC(c->prm_dev, sizeof(SampleParams));
    if (cudaMallocHost(&c->prm_pinned, sizeof(SampleParams)) != cudaSuccess) {
        c->prm_pinned = nullptr;
        c->fail(DFLASH_E_NOMEM, "pinned host allocation failed");
        return bail(DFLASH_E_NOMEM);
    }
    *c->prm_pinned = SampleParams{1.f, 1.f, 1.f, 0};  // no filter
    if (cudaMemcpyAsync(c->prm_dev, c->prm_pinned, sizeof(SampleParams), cudaMemcpyHostToDevice, c->stream) !=
        cudaSuccess) {
        c->fail(DFLASH_E_CUDA, "copy of the sampling settings failed");
        return bail(DFLASH_E_CUDA);
    }
    ALLOC(c->tokens, R * 4);
    ALLOC(c->row_seq, R * 4);
    ALLOC(c->row_pos, R * 4);
    ALLOC(c->ctx_row_seq, (size_t)rb * 4);
    ALLOC(c->ctx_row_pos, (size_t)rb * 4);
    ALLOC(c->n, (size_t)cfg->max_batch * 4);
    ALLOC(c->anchor, (size_t)cfg->max_batch * 4);
    ALLOC(c->proposal, (size_t)cfg->max_batch * c->Bmax * 4);
    ALLOC(c->posterior, (size_t)rb * 4);
    ALLOC(c->argbuf, (size_t)rb * 4);
    ALLOC(c->keys, (size_t)std::max(rb, cfg->max_batch) * 8);
    ALLOC(c->accepted, (size_t)cfg->max_batch * 4);
    ALLOC(c->bonus, (size_t)cfg->max_batch * 4);
    ALLOC(c->drafts, (size_t)cfg->max_batch * c->Bmax * 4);
    ALLOC(c->errw, 16);
    ALLOC(c->attn_ws, ATTN_WS_BYTES);
    ALLOC(c->gemm_ws, GEMM_WS_BYTES);
    ALLOC(c->gemm_counters, (size_t)GEMM_COUNTERS * 4);
    ALLOC(c->gemm_ws_side, GEMM_WS_BYTES);
    ALLOC(c->gemm_counters_side, (size_t)GEMM_COUNTERS * 4);
    if (cfg->flags & DFLASH_FLAG_KEEP_LOGITS) {
        ALLOC(c->keep_prefill, (size_t)cfg->max_batch * V * 4);
        ALLOC(c->keep_draft, (size_t)rb * V * 4);
        ALLOC(c->keep_verify, (size_t)rb * V * 4);
        ALLOC(c->keep_hidden, (size_t)rb * d * 4);
    }
    // caches start at zero: attention stages whole 64-token pages, so slots past
    // a sequence's length must hold finite values
    if (cudaMemsetAsync(c->tK, 0, (size_t)c->Lt * c->kv.layer_stride * esz, c->stream) != cudaSuccess ||
        cudaMemsetAsync(c->tV, 0, (size_t)c->Lt * c->kv.layer_stride * esz, c->stream) != cudaSuccess ||
        cudaMemsetAsync(c->dK, 0, (size_t)c->Ld * c->kv.layer_stride * esz, c->stream) != cudaSuccess ||
        cudaMemsetAsync(c->dV, 0, (size_t)c->Ld * c->kv.layer_stride * esz, c->stream) != cudaSuccess ||
        cudaMemsetAsync(c->errw, 0, 16, c->stream) != cudaSuccess ||
        cudaMemsetAsync(c->gemm_counters, 0, (size_t)GEMM_COUNTERS * 4, c->stream) != cudaSuccess ||
        cudaMemsetAsync(c->gemm_counters_side, 0, (size_t)GEMM_COUNTERS * 4, c->stream) != cudaSuccess ||
        cudaMemsetAsync(c->n, 0, (size_t)cfg->max_batch * 4, c->stream) != cudaSuccess) {
        c->fail(DFLASH_E_CUDA, "memset failed");
        return bail(DFLASH_E_CUDA);
    }
    for (int i = 0; i < 4; ++i)
        if (cudaEventCreate(&c->ev[i]) != cudaSuccess) {
            c->fail(DFLASH_E_CUDA, "event creation failed");
            return bail(DFLASH_E_CUDA);
        }
    c->events = true;
    if (cudaStreamCreateWithFlags(&c->cap_stream, cudaStreamNonBlocking) != cudaSuccess) {
        c->fail(DFLASH_E_CUDA, "stream creation failed");
        return bail(DFLASH_E_CUDA);
    }
    if (cudaStreamCreateWithFlags(&c->side_stream, cudaStreamNonBlocking) != cudaSuccess) {
        c->fail(DFLASH_E_CUDA, "stream creation failed");
        return bail(DFLASH_E_CUDA);
    }
    c->ctx_ev.assign(c->Ld + 1, nullptr);
    for (auto& e : c->ctx_ev)
        if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) {
            e = nullptr;
            c->fail(DFLASH_E_CUDA, "event creation failed");
            return bail(DFLASH_E_CUDA);
        }
    c->graphs = (cfg->flags & DFLASH_FLAG_NO_GRAPHS) == 0;
    memset(c->prof_acc, 0, sizeof c->prof_acc);
    if ((cfg->flags & DFLASH_FLAG_PROFILE) && dflash_set_profiling(c, 1) != DFLASH_OK) return bail(DFLASH_E_CUDA);
    if (cudaStreamSynchronize(c->stream) != cudaSuccess) {
        c->fail(DFLASH_E_CUDA, "weight packing failed: %s", cudaGetErrorString(cudaGetLastError()));
        return bail(DFLASH_E_CUDA);
    }
#undef ALLOC
    *out = c;
    return DFLASH_OK;
}

dflash_status dflash_prefill(dflash_ctx* c, int32_t batch, const int32_t* lens, const int32_t* toks, int32_t* first) {
    if (!c) return DFLASH_E_INVAL;
    if (batch < 1 || batch > c->cfg.max_batch) return c->fail(DFLASH_E_INVAL, "batch %d outside [1, %d]", batch, c->cfg.max_batch);
    if (!lens || !toks || !first) return c->fail(DFLASH_E_INVAL, "NULL argument");
    size_t total = 0;
    for (int s = 0; s < batch; ++s) {
        if (lens[s] < 1) return c->fail(DFLASH_E_INVAL, "prompt %d has length %d", s, lens[s]);
        if (lens[s] + c->B > c->cfg.max_seq_len)
            return c->fail(DFLASH_E_CAPACITY, "prompt %d: length %d + block %d exceeds max_seq_len %d", s, lens[s],
                           c->B, c->cfg.max_seq_len);
        total += lens[s];
    }
    for (size_t i = 0; i < total; ++i)
        if (toks[i] < 0 || toks[i] >= c->V) return c->fail(DFLASH_E_INVAL, "prompt token %zu = %d outside [0, %d)", i, toks[i], c->V);
    // a new batch: every page returns to the pool, then each prompt (+ one block) takes its own
    pool_reset(c);
    for (int s = 0; s < batch; ++s)
        if (!pool_ensure(c, s, (long long)lens[s] + c->B)) {
            const dflash_status st = pool_full(c, s, (long long)lens[s] + c->B);
            pool_reset(c);
            c->batch = 0;
            c->state = ST_EMPTY;
            const dflash_status up = pool_upload(c);
            return up ? up : st;
        }
    {
        dflash_status st = pool_upload(c);
        if (st) return st;
    }
    c->batch = batch;
    c->state = ST_EMPTY;
    c->pending_append = false;
    c->n_upper.assign(lens, lens + batch);
    if (c->events) cudaEventRecord(c->ev[0], c->stream);
    dflash_status s = c->cfg.dtype == DFLASH_DTYPE_BF16 ? Pass<bf16>{c}.prefill(batch, lens, toks, first)
                                                        : Pass<float>{c}.prefill(batch, lens, toks, first);
    if (s != DFLASH_OK) return s;
    if (c->events) {
        cudaEventRecord(c->ev[1], c->stream);
        cudaEventSynchronize(c->ev[1]);
        float ms = 0.f;
        cudaEventElapsedTime(&ms, c->ev[0], c->ev[1]);
        c->stats.prefill_ms += ms;
    }
    c->state = ST_READY;
    return DFLASH_OK;
}

dflash_status dflash_set_block_size(dflash_ctx* c, int32_t block_size) {
    if (!c) return DFLASH_E_INVAL;
    if (block_size < 1 || block_size > c->Bmax)
        return c->fail(DFLASH_E_INVAL, "block size %d outside [1, %d] (the configured block size)", block_size, c->Bmax);
    if (c->state == ST_DRAFTED) return c->fail(DFLASH_E_STATE, "set_block_size between draft_block and verify");
    c->B = block_size;
    return DFLASH_OK;
}

int32_t dflash_block_size(const dflash_ctx* c) { return c ? c->B : -1; }

dflash_status dflash_set_sampling_filter(dflash_ctx* c, int32_t top_k, float top_p) {
    if (!c) return DFLASH_E_INVAL;
    if (top_k < 0) return c->fail(DFLASH_E_INVAL, "top_k %d is negative", top_k);
    if (!(top_p > 0.f && top_p <= 1.f)) return c->fail(DFLASH_E_INVAL, "top_p %g outside (0, 1]", top_p);
    if (c->state == ST_DRAFTED) return c->fail(DFLASH_E_STATE, "set_sampling_filter between a draft and its verify");
    if (c->top_k == top_k && c->top_p == top_p) return DFLASH_OK;
    CUDA_TRY(c, cudaStreamSynchronize(c->stream));  // an earlier copy from the staging buffer is done
    c->prm_pinned->top_p = top_p;
    c->prm_pinned->top_k = top_k;
    CUDA_TRY(c, cudaMemcpyAsync(&c->prm_dev->top_p, &c->prm_pinned->top_p, 8, cudaMemcpyHostToDevice, c->stream));
    c->top_k = top_k;
    c->top_p = top_p;
    return DFLASH_OK;
}

dflash_status dflash_draft_block(dflash_ctx* c, int32_t* draft_tokens) {
    if (!c) return DFLASH_E_INVAL;
    if (c->state != ST_READY) return c->fail(DFLASH_E_STATE, c->state == ST_EMPTY ? "draft_block before prefill" : "draft_block called twice without verify");
    if (!draft_tokens && c->B > 1) return c->fail(DFLASH_E_INVAL, "draft_tokens is NULL");
    dflash_status s;
    if ((s = capacity_check(c))) return s;
    if ((s = do_draft(c))) return s;
    c->draft_sampled = false;
    bool host = false;
    if (c->B > 1 && draft_tokens != c->drafts)
        if ((s = store_out(c, draft_tokens, c->drafts, (size_t)c->batch * (c->B - 1) * 4, &host))) return s;
    c->state = ST_DRAFTED;
    if (host) return check_device(c);
    return DFLASH_OK;
}

dflash_status dflash_verify(dflash_ctx* c, const int32_t* draft_tokens, int32_t* accepted, int32_t* bonus) {
    if (!c) return DFLASH_E_INVAL;
    if (c->state != ST_DRAFTED) return c->fail(DFLASH_E_STATE, "verify without a preceding draft_block");
    if ((!draft_tokens && c->B > 1) || !accepted || !bonus) return c->fail(DFLASH_E_INVAL, "NULL argument");
    dflash_status s;
    if ((s = load_proposal(c, draft_tokens))) return s;
    if ((s = do_verify(c))) return s;
    c->state = ST_READY;
    bool h1 = false, h2 = false;
    if ((s = store_out(c, accepted, c->accepted, (size_t)c->batch * 4, &h1))) return s;
    if ((s = store_out(c, bonus, c->bonus, (size_t)c->batch * 4, &h2))) return s;
    if (h1) {
        if ((s = check_device(c))) return s;
        for (int i = 0; i < c->batch; ++i) c->n_upper[i] += accepted[i] + 1 - c->B;  // now exact
    } else if (h2) {
        if ((s = check_device(c))) return s;
    }
    return DFLASH_OK;
}

dflash_status dflash_draft_block_sampled(dflash_ctx* c, float temperature, const float* u_draft,
                                        int32_t* draft_tokens) {
    if (!c) return DFLASH_E_INVAL;
    if (c->state != ST_READY) return c->fail(DFLASH_E_STATE, c->state == ST_EMPTY ? "draft_block_sampled before prefill" : "draft_block_sampled called twice without verify");
    if (c->B > 1 && (!draft_tokens || !u_draft)) return c->fail(DFLASH_E_INVAL, "NULL argument");
    if (!sampling_vocab_ok(c->V)) return c->fail(DFLASH_E_INVAL, "vocabulary %d too large for the sampled round", c->V);
    dflash_status s;
    if ((s = set_temperature(c, 0, temperature))) return s;
    if ((s = load_uniforms(c, c->u_draft, u_draft, (size_t)c->batch * (c->B - 1)))) return s;
    if ((s = capacity_check(c))) return s;
    if ((s = do_draft(c, true))) return s;
    c->draft_sampled = true;
    bool host = false;
    if (c->B > 1 && draft_tokens != c->drafts)
        if ((s = store_out(c, draft_tokens, c->drafts, (size_t)c->batch * (c->B - 1) * 4, &host))) return s;
    c->state = ST_DRAFTED;
    if (host) return check_device(c);
    return DFLASH_OK;
}

dflash_status dflash_verify_sampled(dflash_ctx* c, float temperature, const int32_t* draft_tokens,
                                    const float* u_verify, int32_t* accepted, int32_t* emitted) {
    if (!c) return DFLASH_E_INVAL;
    if (c->state != ST_DRAFTED || (!c->draft_sampled && c->B > 1))
        return c->fail(DFLASH_E_STATE, "verify_sampled needs a preceding draft_block_sampled");
    if ((!draft_tokens && c->B > 1) || !u_verify || !accepted || !emitted) return c->fail(DFLASH_E_INVAL, "NULL argument");
    if (!sampling_vocab_ok(c->V)) return c->fail(DFLASH_E_INVAL, "vocabulary %d too large for the sampled round", c->V);
    dflash_status s;
    if ((s = set_temperature(c, 1, temperature))) return s;
    if ((s = load_uniforms(c, c->u_verify, u_verify, (size_t)c->batch * c->B))) return s;
    if ((s = load_proposal(c, draft_tokens))) return s;
    if ((s = do_verify(c, true))) return s;
    c->state = ST_READY;
    bool h1 = false, h2 = false;
    if ((s = store_out(c, accepted, c->accepted, (size_t)c->batch * 4, &h1))) return s;
    if ((s = store_out(c, emitted, c->bonus, (size_t)c->batch * 4, &h2))) return s;
    if (h1) {
        if ((s = check_device(c))) return s;
        for (int i = 0; i < c->batch; ++i) c->n_upper[i] += accepted[i] + 1 - c->B;  // now exact
    } else if (h2) {
        if ((s = check_device(c))) return s;
    }
    return DFLASH_OK;
}

dflash_status dflash_train_forward(dflash_ctx* c, int32_t n_tokens, const int32_t* tokens, int32_t n_anchors,
                                   const int32_t* anchors, float lambda, float* loss) {
    if (!c) return DFLASH_E_INVAL;
    if (!tokens || !anchors || !loss || n_anchors < 1) return c->fail(DFLASH_E_INVAL, "NULL argument or no anchors");
    const int B = c->B, m = n_anchors;
    if (B < 2) return c->fail(DFLASH_E_INVAL, "block size 1 predicts no token");
    if (!(lambda > 0.f) || !std::isfinite(lambda)) return c->fail(DFLASH_E_INVAL, "lambda %g is not positive", lambda);
    if (m + 1 > c->cfg.max_batch)
        return c->fail(DFLASH_E_CAPACITY, "%d anchors need max_batch >= %d", m, m + 1);
    for (int i = 0; i < m; ++i)
        if (anchors[i] < 1 || anchors[i] + B - 1 >= n_tokens)
            return c->fail(DFLASH_E_INVAL, "anchor %d = %d outside [1, %d]", i, anchors[i], n_tokens - B);
    // 1. the target's features of the clean sequence: its context K/V in slot 0
    int first = 0;
    dflash_status s = dflash_prefill(c, 1, &n_tokens, tokens, &first);
    if (s) return s;
    // 2. slot i+1 shares slot 0's pages below its anchor's page and takes its own pages from the
    //    pool for the rest of its block
    for (int i = 0; i < m; ++i) {
        const int p0 = anchors[i] >> PAGE_SHIFT;
        c->pool.share(i + 1, 0, p0);
        if (!pool_ensure(c, i + 1, (long long)anchors[i] + B)) {
            const dflash_status st = pool_full(c, i + 1, (long long)anchors[i] + B);
            pool_reset(c);
            c->batch = 0;
            c->state = ST_EMPTY;
            const dflash_status up = pool_upload(c);
            return up ? up : st;
        }
    }
    if ((s = pool_upload(c))) return s;
    // 3. its own copy of the anchor's page (the context rows below the anchor in that page)
    const size_t page_elems = (size_t)c->Hkv * PAGE_TOKENS * c->hd;
    for (int l = 0; l < c->Ld; ++l)
        for (int i = 0; i < m; ++i) {
            const int p0 = anchors[i] >> PAGE_SHIFT;
            const size_t src = (size_t)l * c->kv.layer_stride + (size_t)c->pool.page(0, p0) * page_elems;
            const size_t dst =
                (size_t)l * c->kv.layer_stride + (size_t)c->pool.page(i + 1, p0) * page_elems;
            CUDA_TRY(c, cudaMemcpyAsync((char*)c->dK + dst * c->esz, (char*)c->dK + src * c->esz, page_elems * c->esz,
                                        cudaMemcpyDeviceToDevice, c->stream));
            CUDA_TRY(c, cudaMemcpyAsync((char*)c->dV + dst * c->esz, (char*)c->dV + src * c->esz, page_elems * c->esz,
                                        cudaMemcpyDeviceToDevice, c->stream));
        }
    // 4. one block per anchor: slot i+1 has length a_i and anchor token x[a_i]; labels x[a_i + k]
    std::vector<int> nh(m + 1), ah(m + 1), labels((size_t)m * (B - 1));
    nh[0] = n_tokens;
    ah[0] = first;
    for (int i = 0; i < m; ++i) {
        nh[i + 1] = anchors[i];
        ah[i + 1] = tokens[anchors[i]];
        for (int k = 1; k < B; ++k) labels[(size_t)i * (B - 1) + k - 1] = tokens[anchors[i] + k];
    }
    CUDA_TRY(c, cudaMemcpyAsync(c->n, nh.data(), nh.size() * 4, cudaMemcpyHostToDevice, c->stream));
    CUDA_TRY(c, cudaMemcpyAsync(c->anchor, ah.data(), ah.size() * 4, cudaMemcpyHostToDevice, c->stream));
    CUDA_TRY(c, cudaMemcpyAsync(c->proposal, labels.data(), labels.size() * 4, cudaMemcpyHostToDevice, c->stream));
    c->batch = m + 1;
    c->n_upper = nh;
    c->pending_append = false;
    // 5. the drafter over every block at once, logits kept; 6. per-row cross-entropy
    c->draft_logits_out = true;
    if (c->cfg.dtype == DFLASH_DTYPE_BF16) Pass<bf16>{c}.draft();
    else Pass<float>{c}.draft();
    c->draft_logits_out = false;
    {
        Launch L = c->L();
        row_nll(L, c->dlogits, c->V, B, 1, m, c->proposal, c->u_draft);
    }
    std::vector<float> nll((size_t)m * (B - 1));
    CUDA_TRY(c, cudaMemcpyAsync(nll.data(), c->u_draft, nll.size() * 4, cudaMemcpyDeviceToHost, c->stream));
    // 7. every page back to the pool; the session needs a new prefill before any round
    pool_reset(c);
    if ((s = pool_upload(c))) return s;
    CUDA_TRY(c, cudaStreamSynchronize(c->stream));
    c->batch = 0;
    c->state = ST_EMPTY;
    if ((s = launch_check(c))) return s;
    if ((s = check_device(c))) return s;
    // eq. 12: mean over anchors of the exp(-(k-1)/lambda)-weighted sum, in a fixed order
    double total = 0.0;
    for (int i = 0; i < m; ++i) {
        double blk = 0.0;
        for (int k = 1; k < B; ++k) blk += exp(-(double)(k - 1) / (double)lambda) * (double)nll[(size_t)i * (B - 1) + k - 1];
        total += blk;
    }
    *loss = (float)(total / m);
    return DFLASH_OK;
}

dflash_status dflash_generate(dflash_ctx* c, int32_t batch, const int32_t* lens, const int32_t* toks, int32_t N,
                              int32_t* out_tokens, int32_t* out_lens, dflash_stats* stats) {
    if (!c) return DFLASH_E_INVAL;
    if (N < 1 || !out_tokens || !out_lens) return c->fail(DFLASH_E_INVAL, "max_new_tokens < 1 or NULL output");
    dflash_status s;
    std::vector<int> first(batch > 0 ? batch : 1);
    if ((s = dflash_prefill(c, batch, lens, toks, first.data()))) return s;
    const int B = c->B;
    std::vector<int> cnt(batch, 0), acc(batch), bon(batch), dr((size_t)batch * (B > 1 ? B - 1 : 1));
    for (int i = 0; i < batch; ++i) {
        out_tokens[(size_t)i * N] = first[i];
        cnt[i] = 1;
    }
    c->stats.tokens += batch;
    auto done = [&]() {
        for (int i = 0; i < batch; ++i)
            if (cnt[i] < N) return false;
        return true;
    };
    while (!done()) {
        cudaEventRecord(c->ev[0], c->stream);
        if ((s = dflash_draft_block(c, c->drafts))) return s;
        cudaEventRecord(c->ev[1], c->stream);
        if ((s = dflash_verify(c, c->drafts, c->accepted, c->bonus))) return s;
        cudaEventRecord(c->ev[2], c->stream);
        CUDA_TRY(c, cudaMemcpyAsync(acc.data(), c->accepted, (size_t)batch * 4, cudaMemcpyDeviceToHost, c->stream));
        CUDA_TRY(c, cudaMemcpyAsync(bon.data(), c->bonus, (size_t)batch * 4, cudaMemcpyDeviceToHost, c->stream));
        if (B > 1)
            CUDA_TRY(c, cudaMemcpyAsync(dr.data(), c->proposal, (size_t)batch * (B - 1) * 4, cudaMemcpyDeviceToHost,
                                        c->stream));
        if ((s = check_device(c))) return s;
        float t1 = 0.f, t2 = 0.f;
        cudaEventElapsedTime(&t1, c->ev[0], c->ev[1]);
        cudaEventElapsedTime(&t2, c->ev[1], c->ev[2]);
        c->stats.draft_ms += t1;
        c->stats.verify_ms += t2;
        c->stats.rounds += 1;
        for (int i = 0; i < batch; ++i) {
            c->n_upper[i] += acc[i] + 1 - B;
            c->stats.accepted += acc[i];
            for (int j = 0; j < acc[i] && cnt[i] < N; ++j) out_tokens[(size_t)i * N + cnt[i]++] = dr[(size_t)i * (B - 1) + j];
            if (cnt[i] < N) out_tokens[(size_t)i * N + cnt[i]++] = bon[i];
            c->stats.tokens += acc[i] + 1;
        }
        bool room = true;
        for (int i = 0; i < batch; ++i)
            if (cnt[i] < N && c->n_upper[i] + B > c->cfg.max_seq_len) room = false;
        if (!room) return c->fail(DFLASH_E_CAPACITY, "max_seq_len too small for max_new_tokens");
    }
    for (int i = 0; i < batch; ++i) out_lens[i] = N;
    c->stats.kernel_launches = c->launches;
    if (stats) *stats = c->stats;
    return DFLASH_OK;
}

dflash_status dflash_inspect(dflash_ctx* c, int32_t what, int32_t seq, int32_t layer, void* dst, size_t bytes,
                             size_t* written) {
    if (!c || !dst) return DFLASH_E_INVAL;
    size_t need = 0;
    const int b = c->batch, B = c->B;
    auto simple = [&](const void* p, size_t n) -> dflash_status {
        if (bytes < n) return c->fail(DFLASH_E_INVAL, "buffer of %zu bytes, need %zu", bytes, n);
        if (!p) return c->fail(DFLASH_E_INVAL, "item not kept (set DFLASH_FLAG_KEEP_LOGITS)");
        CUDA_TRY(c, cudaMemcpyAsync(dst, p, n, cudaMemcpyDeviceToHost, c->stream));
        CUDA_TRY(c, cudaStreamSynchronize(c->stream));
        if (written) *written = n;
        return DFLASH_OK;
    };
    switch (what) {
        case DFLASH_INSPECT_LENGTHS: return simple(c->n, (size_t)b * 4);
        case DFLASH_INSPECT_ANCHORS: return simple(c->anchor, (size_t)b * 4);
        case DFLASH_INSPECT_POSTERIOR: return simple(c->posterior, (size_t)b * B * 4);
        case DFLASH_INSPECT_LOGITS_PREFILL: return simple(c->keep_prefill, (size_t)b * c->V * 4);
        case DFLASH_INSPECT_LOGITS_DRAFT: return simple(c->keep_draft, (size_t)b * B * c->V * 4);
        case DFLASH_INSPECT_LOGITS_VERIFY: return simple(c->keep_verify, (size_t)b * B * c->V * 4);
        case DFLASH_INSPECT_HIDDEN_VERIFY: return simple(c->keep_hidden, (size_t)b * B * c->d * 4);
        case DFLASH_INSPECT_PROFILE: {
            if (bytes < sizeof(c->prof_acc)) return c->fail(DFLASH_E_INVAL, "buffer too small");
            dflash_status s = prof_drain(c);
            if (s) return s;
            memcpy(dst, c->prof_acc, sizeof(c->prof_acc));
            if (written) *written = sizeof(c->prof_acc);
            return DFLASH_OK;
        }
        case DFLASH_INSPECT_PROFILE_RESET: {
            dflash_status s = prof_drain(c);
            if (s) return s;
            memset(c->prof_acc, 0, sizeof(c->prof_acc));
            if (written) *written = 0;
            return DFLASH_OK;
        }
        case DFLASH_INSPECT_STATS: {
            if (bytes < sizeof(dflash_stats)) return c->fail(DFLASH_E_INVAL, "buffer too small");
            c->stats.kernel_launches = c->launches;
            memcpy(dst, &c->stats, sizeof(dflash_stats));
            if (written) *written = sizeof(dflash_stats);
            return DFLASH_OK;
        }
        case DFLASH_INSPECT_TARGET_K:
        case DFLASH_INSPECT_TARGET_V:
        case DFLASH_INSPECT_DRAFT_K:
        case DFLASH_INSPECT_DRAFT_V: {
            const bool tgt = what == DFLASH_INSPECT_TARGET_K || what == DFLASH_INSPECT_TARGET_V;
            const int nl = tgt ? c->Lt : c->Ld;
            if (seq < 0 || seq >= b || layer < 0 || layer >= nl) return c->fail(DFLASH_E_INVAL, "seq/layer out of range");
            int ns = 0;
            CUDA_TRY(c, cudaMemcpyAsync(&ns, c->n + seq, 4, cudaMemcpyDeviceToHost, c->stream));
            CUDA_TRY(c, cudaStreamSynchronize(c->stream));
            need = (size_t)ns * c->kvd * c->esz;
            if (bytes < need) return c->fail(DFLASH_E_INVAL, "buffer of %zu bytes, need %zu", bytes, need);
            void* base = (what == DFLASH_INSPECT_TARGET_K) ? c->tK : (what == DFLASH_INSPECT_TARGET_V) ? c->tV
                       : (what == DFLASH_INSPECT_DRAFT_K) ? c->dK : c->dV;
            std::vector<int> pt(c->kv.pages_per_seq);
            CUDA_TRY(c, cudaMemcpy(pt.data(), c->page_table + (size_t)seq * c->kv.pages_per_seq, pt.size() * 4,
                                   cudaMemcpyDeviceToHost));
            const size_t page_elems = (size_t)c->Hkv * PAGE_TOKENS * c->hd;
            std::vector<char> page(page_elems * c->esz);
            char* o = (char*)dst;
            for (int p0 = 0; p0 < ns; p0 += PAGE_TOKENS) {
                const char* src_page = (const char*)base +
                    ((size_t)layer * c->kv.layer_stride + (size_t)pt[p0 / PAGE_TOKENS] * page_elems) * c->esz;
                CUDA_TRY(c, cudaMemcpy(page.data(), src_page, page.size(), cudaMemcpyDeviceToHost));
                for (int t = p0; t < std::min(ns, p0 + PAGE_TOKENS); ++t)
                    for (int h = 0; h < c->Hkv; ++h)
                        memcpy(o + ((size_t)t * c->Hkv + h) * c->hd * c->esz,
                               page.data() + (((size_t)h * PAGE_TOKENS) + (t - p0)) * c->hd * c->esz, c->hd * c->esz);
            }
            if (written) *written = need;
            return DFLASH_OK;
        }
        default: return c->fail(DFLASH_E_INVAL, "unknown inspect item %d", what);
    }
}

dflash_status dflash_set_profiling(dflash_ctx* c, int32_t on) {
    if (!c) return DFLASH_E_INVAL;
    if (on && c->prof_ev.empty()) {
        c->prof_ev.resize(4096);
        for (auto& e : c->prof_ev) CUDA_TRY(c, cudaEventCreate(&e));
    }
    if (!on) {
        dflash_status s = prof_drain(c);
        if (s) return s;
    }
    c->profiling = on != 0;
    return DFLASH_OK;
}

void dflash_destroy(dflash_ctx* c) {
    if (!c) return;
    if (c->stream) cudaStreamSynchronize(c->stream);
    else cudaDeviceSynchronize();
    for (void* p : c->allocs) {
        if (c->cfg.free) c->cfg.free(p, c->cfg.alloc_user);
        else cudaFree(p);
    }
    if (c->events)
        for (int i = 0; i < 4; ++i) cudaEventDestroy(c->ev[i]);
    for (auto& e : c->prof_ev) cudaEventDestroy(e);
    reset_graph(c->g_draft[0]);
    reset_graph(c->g_draft[1]);
    reset_graph(c->g_verify);
    reset_graph(c->g_draft_s[0]);
    reset_graph(c->g_draft_s[1]);
    reset_graph(c->g_verify_s);
    if (c->cap_stream) cudaStreamDestroy(c->cap_stream);
    for (auto& e : c->ctx_ev)
        if (e) cudaEventDestroy(e);
    if (c->side_stream) cudaStreamDestroy(c->side_stream);
    if (c->prm_pinned) cudaFreeHost(c->prm_pinned);
    delete c;
}

const char* dflash_last_error(const dflash_ctx* c) {
    return c ? c->err.c_str() : g_init_error.c_str();
}

}  // extern "C"
