// Allocation-free variant of the shared-head argmax (see
// dflash_head_argmax_noalloc in include/dflash.h).
//
// Some callers cannot allocate device memory at all: code that runs inside
// another framework's memory pool, an embedded runtime whose allocator is
// locked, or a process whose memory budget is fixed before this library
// loads.  For them the head's two intermediates - the normalised rows and the
// fp32 logits - live in one file-scope device array of fixed size instead of
// buffers from cudaMalloc or a caller's allocator.  Every GPU that loads this
// library holds that array until the process exits.
#include <stdio.h>

#include <mutex>

#include "dflash.h"
#include "launch.h"

using namespace dfl;

namespace {

constexpr size_t NOALLOC_SCRATCH_BYTES = (size_t)DFLASH_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_head_scratch[NOALLOC_SCRATCH_BYTES];

constexpr int MAX_DEVICES = 64;
std::mutex g_mu;
void* g_scratch_addr[MAX_DEVICES] = {};

// Device address of g_head_scratch on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device with that device current.
cudaError_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= MAX_DEVICES) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_head_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

dflash_status fail(dflash_status s, const char* msg) {
    dfl::set_global_error(msg);  // readable through dflash_last_error(NULL)
    return s;
}

// out[r] = -1 for every row when a bounded device-side wait of this call ran out
// (the error word is cleared at the start of each call).
__global__ void poison_on_error_kernel(const uint32_t* __restrict__ err, int rows, int* __restrict__ out) {
    if (*err == 0u) return;
    for (int r = blockIdx.x * blockDim.x + threadIdx.x; r < rows; r += gridDim.x * blockDim.x) out[r] = -1;
}

// Queues the norm, the head GEMM, the row argmax and the error check; false when a
// kernel could not be prepared (for example a tensor map that could not be encoded).
template <typename T>
bool run_head(const float* x, const float* norm_w, float eps, const void* head, int rows, int d, int vocab, int* out,
              unsigned char* scratch, cudaStream_t stream) {
    bool failed = false;
    Launch L{stream, nullptr};
    L.failed = &failed;
    uint32_t* err = reinterpret_cast<uint32_t*>(scratch);  // first 256 bytes: device error word
    L.err = err;
    if (cudaMemsetAsync(err, 0, sizeof(uint32_t), stream) != cudaSuccess) return false;
    scratch += 256;
    T* xn = reinterpret_cast<T*>(scratch);
    const size_t xn_bytes = ((size_t)rows * d * sizeof(T) + 255) / 256 * 256;
    float* logits = reinterpret_cast<float*>(scratch + xn_bytes);
    rmsnorm_rows<T>(L, x, d, norm_w, rows, d, eps, xn, d);
    gemm<T>(L, xn, d, reinterpret_cast<const T*>(head), rows, vocab, d, logits, vocab, false);
    argmax_rows(L, logits, vocab, rows, vocab, out);
    launch_k(L, poison_on_error_kernel, dim3((rows + 255) / 256), dim3(256), 0, 1, (const uint32_t*)err, rows, out);
    return !failed;
}

}  // namespace

extern "C" dflash_status dflash_head_argmax_noalloc(int32_t dtype, const float* x, const float* norm_w, float eps,
                                                     const void* head, int32_t rows, int32_t d_model, int32_t vocab,
                                                     int32_t* out, void* cuda_stream) {
    if (!x || !norm_w || !head || !out) return fail(DFLASH_E_INVAL, "NULL pointer argument");
    if (dtype != DFLASH_DTYPE_F32 && dtype != DFLASH_DTYPE_BF16) return fail(DFLASH_E_INVAL, "dtype must be F32 or BF16");
    if (rows < 1 || d_model < 8 || d_model % 8 || vocab < 1 || !(eps > 0.f))
        return fail(DFLASH_E_INVAL, "rows >= 1, d_model a positive multiple of 8, vocab >= 1 and eps > 0 required");
    // the head is read through TMA (bf16) and both matrices with 16-byte vector loads
    if (((uintptr_t)x | (uintptr_t)head | (uintptr_t)norm_w) & 15u)
        return fail(DFLASH_E_INVAL, "x, norm_w and head must be 16-byte aligned");
    const size_t esz = dtype == DFLASH_DTYPE_BF16 ? 2 : 4;
    const size_t need = 256 + ((size_t)rows * d_model * esz + 255) / 256 * 256 + (size_t)rows * vocab * 4;
    if (need > NOALLOC_SCRATCH_BYTES) {
        char buf[256];
        snprintf(buf, sizeof buf,
                 "rows x (d_model x %zu + vocab x 4) needs %zu bytes of scratch; the fixed maximum is %zu bytes",
                 esz, need, NOALLOC_SCRATCH_BYTES);
        return fail(DFLASH_E_INVAL, buf);
    }
    void* scratch = nullptr;
    cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess) return fail(DFLASH_E_CUDA, cudaGetErrorString(e));
    cudaStream_t s = (cudaStream_t)cuda_stream;
    const bool queued =
        dtype == DFLASH_DTYPE_BF16
            ? run_head<bf16>(x, norm_w, eps, head, rows, d_model, vocab, out, (unsigned char*)scratch, s)
            : run_head<float>(x, norm_w, eps, head, rows, d_model, vocab, out, (unsigned char*)scratch, s);
    e = cudaGetLastError();
    if (e != cudaSuccess) return fail(DFLASH_E_CUDA, cudaGetErrorString(e));
    if (!queued) return fail(DFLASH_E_CUDA, "a kernel of the head could not be prepared (tensor map or launch setup)");
    return DFLASH_OK;
}
