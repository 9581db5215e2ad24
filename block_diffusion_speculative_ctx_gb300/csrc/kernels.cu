// Row-wise kernels of the round: embedding gather, RMSNorm, per-head q/k norm
// with RoPE and KV-cache store, SwiGLU product, context-layer capture, row
// argmax, block construction and greedy acceptance.
#include "launch.h"

namespace dfl {

// ---------------------------------------------------------------- embedding
template <typename T>
__global__ void embed_kernel(const int* __restrict__ tokens, const T* __restrict__ embed, int vocab, int d,
                             float* __restrict__ x, uint32_t* err, float* __restrict__ ss_out, int ss_ld) {
    pdl_wait();
    pdl_trigger();
    __shared__ float part[64][4];  // [128-column tile][quarter]
    const int r = blockIdx.x;
    int t = tokens[r];
    if (t < 0 || t >= vocab) {
        if (threadIdx.x == 0) atomicOr(err, ERR_TOKEN_RANGE);
        t = 0;
    }
    const T* src = embed + (size_t)t * d;
    float* dst = x + (size_t)r * d;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // blockDim 256: in step i, warp w covers columns 256 i + 32 w .. +31, i.e. quarter (w & 3)
    // of tile 2 i + (w >> 2); quarter sums are added in a fixed order below
    for (int c0 = 0; c0 < d; c0 += 256) {
        const int c = c0 + threadIdx.x;
        float v = 0.f;
        if (c < d) {
            v = to_f32(src[c]);
            dst[c] = v;
        }
        if (ss_out) {
            const float sq = warp_sum(v * v);
            if (lane == 0) part[(c0 >> 7) + (warp >> 2)][warp & 3] = sq;
        }
    }
    if (ss_out) {
        __syncthreads();
        const int tiles = (d + 127) / 128;
        if (threadIdx.x < tiles)
            ss_out[(size_t)threadIdx.x * ss_ld + r] =
                ((part[threadIdx.x][0] + part[threadIdx.x][1]) + part[threadIdx.x][2]) + part[threadIdx.x][3];
    }
}

template <typename T>
void embed_rows(const Launch& L, const int* tokens, const T* embed, int vocab, int d, int rows, float* x,
                uint32_t* err, float* ss_out, int ss_ld) {
    if (rows <= 0) return;
    launch_k(L, embed_kernel<T>, dim3(rows), dim3(256), 0, 1, tokens, embed, vocab, d, x, err, ss_out, ss_ld);
}

// ------------------------------------------------------------------ RMSNorm
// out = x / sqrt(mean(x^2) + eps) * w, one CTA per row.
template <typename T>
__global__ void rmsnorm_kernel(const float* __restrict__ x, int ldx, const int* __restrict__ row_idx,
                               const float* __restrict__ w, int d, float eps, T* __restrict__ out, int ldo) {
    pdl_wait();
    pdl_trigger();
    __shared__ float red[32];
    const int r = blockIdx.x;
    const int src_row = row_idx ? row_idx[r] : r;
    const float* xr = x + (size_t)src_row * ldx;
    float ss = 0.f;
    for (int c = threadIdx.x; c < d; c += blockDim.x) {
        float v = xr[c];
        ss += v * v;
    }
    ss = block_sum(ss, red);
    const float inv = rsqrtf(ss / (float)d + eps);
    T* o = out + (size_t)r * ldo;
    for (int c = threadIdx.x; c < d; c += blockDim.x) o[c] = from_f32<T>(xr[c] * inv * w[c]);
}

template <typename T>
void rmsnorm_rows(const Launch& L, const float* x, int ldx, const float* w, int rows, int d, float eps, T* out,
                  int ldo) {
    if (rows <= 0) return;
    launch_k(L, rmsnorm_kernel<T>, dim3(rows), dim3(256), 0, 1, x, ldx, (const int*)nullptr, w, d, eps, out, ldo);
}

template <typename T>
void rmsnorm_gather(const Launch& L, const float* x, int ldx, const int* row_idx, const float* w, int rows, int d,
                    float eps, T* out, int ldo) {
    if (rows <= 0) return;
    launch_k(L, rmsnorm_kernel<T>, dim3(rows), dim3(256), 0, 1, x, ldx, row_idx, w, d, eps, out, ldo);
}

// ------------------------------------------------- q/k norm, RoPE, KV store
// One CTA per row, one warp per head (query heads, then key heads, then value
// heads).  Lane l holds elements l + 32 i of the head; the rotary pair of
// element j is j + hd/2, i.e. the same lane at i + hd/64.
template <typename T, int HD>
__global__ void qkv_store_kernel(QKVStore p) {
    pdl_wait();
    pdl_trigger();
    constexpr int PER = HD / 32;    // elements per lane
    constexpr int HALF = PER / 2;   // pair offset in i
    const int r = blockIdx.x;
    const int seq = p.row_seq[r];
    if (seq < 0) return;
    const int pos = p.row_pos[r];
    if (pos < 0 || pos >= p.max_pos) {
        if (threadIdx.x == 0) atomicOr(p.err, ERR_POSITION_RANGE);
        return;
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    const int nq = (p.q_off >= 0) ? p.H : 0;
    const int nheads = nq + 2 * p.Hkv;
    const float* row = p.qkv + (size_t)r * p.ld;
    const float2* rp = p.rope + (size_t)pos * (HD / 2);
    for (int h = warp; h < nheads; h += nwarps) {
        float v[PER];
        int kind, hh;  // 0 = q, 1 = k, 2 = v
        if (h < nq) { kind = 0; hh = h; }
        else if (h < nq + p.Hkv) { kind = 1; hh = h - nq; }
        else { kind = 2; hh = h - nq - p.Hkv; }
        const int col = (kind == 0 ? p.q_off : kind == 1 ? p.k_off : p.v_off) + hh * HD;
#pragma unroll
        for (int i = 0; i < PER; ++i) v[i] = row[col + lane + 32 * i];
        if (kind < 2) {
            const float* nw = (kind == 0) ? p.q_norm : p.k_norm;
            if (nw) {
                float ss = 0.f;
#pragma unroll
                for (int i = 0; i < PER; ++i) ss += v[i] * v[i];
                ss = warp_sum(ss);
                const float inv = rsqrtf(ss / (float)HD + p.eps);
#pragma unroll
                for (int i = 0; i < PER; ++i) v[i] = v[i] * inv * nw[lane + 32 * i];
            }
#pragma unroll
            for (int i = 0; i < HALF; ++i) {
                const float2 cs = rp[lane + 32 * i];
                const float x1 = v[i], x2 = v[i + HALF];
                v[i] = x1 * cs.x - x2 * cs.y;
                v[i + HALF] = x2 * cs.x + x1 * cs.y;
            }
        }
        if (kind == 0) {
            T* q = reinterpret_cast<T*>(p.q_out) + (size_t)r * p.H * HD + hh * HD;
#pragma unroll
            for (int i = 0; i < PER; ++i) q[lane + 32 * i] = from_f32<T>(v[i]);
        } else {
            T* base = reinterpret_cast<T*>(kind == 1 ? p.Kc : p.Vc);
            T* dst = base + kv_offset(p.kv, p.page_table, seq, pos, hh);
#pragma unroll
            for (int i = 0; i < PER; ++i) dst[lane + 32 * i] = from_f32<T>(v[i]);
        }
    }
}

template <typename T>
void qk_norm_rope_store(const Launch& L, const QKVStore& p) {
    if (p.rows <= 0) return;
    const int nheads = (p.q_off >= 0 ? p.H : 0) + 2 * p.Hkv;
    int warps = nheads < 16 ? nheads : 16;
    if (p.hd == 128)
        launch_k(L, qkv_store_kernel<T, 128>, dim3(p.rows), dim3(32 * warps), 0, 1, p);
    else
        launch_k(L, qkv_store_kernel<T, 64>, dim3(p.rows), dim3(32 * warps), 0, 1, p);
}

// -------------------------------------------------------------------- SwiGLU
// gu = [gate | up] per row (2F fp32); out = silu(gate) * up.
template <typename T>
__global__ void silu_mul_kernel(const float* __restrict__ gu, int F, int rows, T* __restrict__ out) {
    pdl_wait();
    pdl_trigger();
    const size_t n = (size_t)rows * F;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const size_t r = i / F, f = i % F;
        const float g = gu[r * 2 * F + f], u = gu[r * 2 * F + F + f];
        out[i] = from_f32<T>(g / (1.f + expf(-g)) * u);
    }
}

template <typename T>
void silu_mul(const Launch& L, const float* gu, int F, int rows, T* out) {
    if (rows <= 0) return;
    size_t n = (size_t)rows * F;
    int blocks = (int)((n + 255) / 256);
    if (blocks > 152 * 16) blocks = 152 * 16;
    launch_k(L, silu_mul_kernel<T>, dim3(blocks), dim3(256), 0, 1, gu, F, rows, out);
}

// ------------------------------------------------------------------ capture
template <typename T>
__global__ void capture_kernel(const float* __restrict__ x, int d, T* __restrict__ stage, int ld, int col) {
    pdl_wait();
    pdl_trigger();
    const int r = blockIdx.x;
    for (int c = threadIdx.x; c < d; c += blockDim.x) stage[(size_t)r * ld + col + c] = from_f32<T>(x[(size_t)r * d + c]);
}

template <typename T>
void capture_rows(const Launch& L, const float* x, int d, int rows, T* stage, int ld_stage, int col) {
    if (rows <= 0) return;
    launch_k(L, capture_kernel<T>, dim3(rows), dim3(256), 0, 1, x, d, stage, ld_stage, col);
}

// ------------------------------------------------------------------- argmax
__global__ void argmax_kernel(const float* __restrict__ logits, long long ld, int V, int* __restrict__ out) {
    pdl_wait();
    pdl_trigger();
    __shared__ unsigned long long red[32];
    const int r = blockIdx.x;
    const float* row = logits + (size_t)r * ld;
    unsigned long long best = 0ull;
    for (int v = threadIdx.x; v < V; v += blockDim.x) {
        unsigned long long k = argmax_key(row[v], (uint32_t)v);
        best = k > best ? k : best;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        unsigned long long t = __shfl_xor_sync(0xffffffffu, best, o);
        best = t > best ? t : best;
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) red[warp] = best;
    __syncthreads();
    if (warp == 0) {
        best = lane < (int)(blockDim.x >> 5) ? red[lane] : 0ull;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            unsigned long long t = __shfl_xor_sync(0xffffffffu, best, o);
            best = t > best ? t : best;
        }
        if (lane == 0) out[r] = (int)argmax_key_index(best);
    }
}

void argmax_rows(const Launch& L, const float* logits, long long ld, int rows, int V, int* out) {
    if (rows <= 0) return;
    launch_k(L, argmax_kernel, dim3(rows), dim3(1024), 0, 1, logits, ld, V, out);
}

__global__ void keys_to_ids_kernel(const unsigned long long* __restrict__ keys, int rows, int block,
                                   int* __restrict__ out) {
    pdl_wait();
    pdl_trigger();
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= rows) return;
    const int id = (int)argmax_key_index(keys[r]);
    if (block <= 0) {
        out[r] = id;
    } else {
        const int j = r % block;
        if (j) out[(r / block) * (block - 1) + j - 1] = id;
    }
}

void keys_to_ids(const Launch& L, const unsigned long long* keys, int rows, int block, int* out) {
    if (rows <= 0) return;
    launch_k(L, keys_to_ids_kernel, dim3((rows + 127) / 128), dim3(128), 0, 1, keys, rows, block, out);
}

// --------------------------------------------------------- round bookkeeping
__global__ void block_rows_kernel(int batch, int B, const int* __restrict__ n, const int* __restrict__ anchor,
                                  const int* __restrict__ proposal, int mask, int vocab, int max_pos,
                                  int* __restrict__ tokens, int* __restrict__ row_seq, int* __restrict__ row_pos,
                                  uint32_t* err) {
    pdl_wait();
    pdl_trigger();
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= batch * B) return;
    const int s = r / B, j = r % B;
    int t;
    if (j == 0) t = anchor[s];
    else if (proposal) t = proposal[s * (B - 1) + j - 1];
    else t = mask;
    if (t < 0 || t >= vocab) {
        atomicOr(err, ERR_TOKEN_RANGE);
        t = 0;
    }
    const int pos = n[s] + j;
    if (pos >= max_pos) atomicOr(err, ERR_POSITION_RANGE);
    tokens[r] = t;
    row_seq[r] = pos < max_pos ? s : -1;
    row_pos[r] = pos;
}

void block_rows(const Launch& L, int batch, int B, const int* n, const int* anchor, const int* proposal, int mask,
                int vocab, int max_pos, int* tokens, int* row_seq, int* row_pos, uint32_t* err) {
    const int rows = batch * B;
    launch_k(L, block_rows_kernel, dim3((rows + 127) / 128), dim3(128), 0, 1, batch, B, n, anchor, proposal, mask,
             vocab, max_pos, tokens, row_seq, row_pos, err);
}

// One thread per sequence: the longest prefix with proposal[j] == posterior[j].
__global__ void accept_kernel(int batch, int B, const int* __restrict__ proposal, const int* __restrict__ posterior,
                              int* __restrict__ n, int* __restrict__ anchor, int* __restrict__ accepted,
                              int* __restrict__ bonus, int* __restrict__ ctx_row_seq, int* __restrict__ ctx_row_pos) {
    pdl_wait();
    pdl_trigger();
    const int s = blockIdx.x * blockDim.x + threadIdx.x;
    if (s >= batch) return;
    const int* d = proposal + (size_t)s * (B - 1);
    const int* post = posterior + (size_t)s * B;
    int a = 0;
    while (a < B - 1 && d[a] == post[a]) ++a;
    const int b = post[a];
    const int n0 = n[s];
    accepted[s] = a;
    bonus[s] = b;
    anchor[s] = b;
    n[s] = n0 + a + 1;
    for (int j = 0; j < B; ++j) {
        ctx_row_seq[s * B + j] = (j <= a) ? s : -1;
        ctx_row_pos[s * B + j] = n0 + j;
    }
}

void accept(const Launch& L, int batch, int B, const int* proposal, const int* posterior, int* n, int* anchor,
            int* accepted, int* bonus, int* ctx_row_seq, int* ctx_row_pos) {
    launch_k(L, accept_kernel, dim3((batch + 63) / 64), dim3(64), 0, 1, batch, B, proposal, posterior, n, anchor,
             accepted, bonus, ctx_row_seq, ctx_row_pos);
}

__global__ void prefill_rows_kernel(int seq, int start, int rows, int* row_seq, int* row_pos) {
    pdl_wait();
    pdl_trigger();
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r < rows) {
        row_seq[r] = seq;
        row_pos[r] = start + r;
    }
}

void fill_prefill_rows(const Launch& L, int seq, int start_pos, int rows, int* row_seq, int* row_pos) {
    launch_k(L, prefill_rows_kernel, dim3((rows + 255) / 256), dim3(256), 0, 1, seq, start_pos, rows, row_seq, row_pos);
}

// ---- explicit instantiations
#define DFL_INST(T)                                                                                         \
    template void embed_rows<T>(const Launch&, const int*, const T*, int, int, int, float*, uint32_t*, float*, \
                                int);                                                                       \
    template void rmsnorm_rows<T>(const Launch&, const float*, int, const float*, int, int, float, T*, int); \
    template void rmsnorm_gather<T>(const Launch&, const float*, int, const int*, const float*, int, int,   \
                                    float, T*, int);                                                        \
    template void qk_norm_rope_store<T>(const Launch&, const QKVStore&);                                    \
    template void silu_mul<T>(const Launch&, const float*, int, int, T*);                                   \
    template void capture_rows<T>(const Launch&, const float*, int, int, T*, int, int);
DFL_INST(float)
DFL_INST(bf16)
#undef DFL_INST

// KV page table entries assigned by the host pool; the updates travel in the kernel's
// parameters, so no host buffer outlives the call.
__global__ void set_pages_kernel(int* __restrict__ table, PageUpdates u) {
    pdl_wait();
    pdl_trigger();
    if ((int)threadIdx.x < u.n) table[u.idx[threadIdx.x]] = u.page[threadIdx.x];
}

void set_pages(const Launch& L, int* table, const PageUpdates& u) {
    if (u.n <= 0) return;
    launch_k(L, set_pages_kernel, dim3(1), dim3(64), 0, 1, table, u);
}

}  // namespace dfl
