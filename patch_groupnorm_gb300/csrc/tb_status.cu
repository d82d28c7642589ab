// tb_status.cu -- the library's device-side status word.
//
// Kernels never trap.  A kernel that meets a condition it cannot complete
// under -- a wait for a tensor copy that runs out of its iteration limit, or,
// in the bounds-checked build, an index outside its tile or output -- records
// a code here (the first one wins) and returns; the host reads the word with
// tb_device_status.  One word per device, in the library's own static device
// memory (nothing is allocated).
#include <mutex>

#include "tb_internal.h"
#include "tileblend.h"

#define TB_API extern "C" __attribute__((visibility("default")))

namespace {

__device__ uint32_t g_status_word = 0;

constexpr int MAX_DEVICES = 64;

// Driver calls reached through the runtime's entry-point query (no driver
// library is linked).
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

struct Cached {
    unsigned long long ctx_id;
    uint32_t* addr;
};
std::mutex g_mu;
Cached g_cache[MAX_DEVICES] = {};

}  // namespace

namespace tb {

// Process-unique id (+1) of the calling thread's current context, 0 if none
// is bound yet or the driver calls are unavailable.
unsigned long long current_context_id() {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(f);
    });
    if (get_current == nullptr || get_id == nullptr) return 0;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
    unsigned long long id = 0;
    if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id + 1;
}

uint32_t* device_status_word() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return nullptr;
    std::lock_guard<std::mutex> lock(g_mu);
    const unsigned long long id = current_context_id();
    Cached& c = g_cache[dev];
    if (c.addr == nullptr || id == 0 || id != c.ctx_id) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) {
            (void)cudaGetLastError();
            return nullptr;
        }
        c.addr = static_cast<uint32_t*>(p);
        c.ctx_id = current_context_id();
    }
    return c.addr;
}

}  // namespace tb

TB_API tb_status tb_device_status(uint32_t* code, int32_t clear) {
    if (code == nullptr) return TB_ERR_NULL;
    uint32_t v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_status_word, sizeof(v));
    if (e != cudaSuccess) {
        tb::record_cuda_error(e);
        return TB_ERR_CUDA;
    }
    *code = v;
    if (clear) {
        const uint32_t zero = 0;
        e = cudaMemcpyToSymbol(g_status_word, &zero, sizeof(zero));
        if (e != cudaSuccess) {
            tb::record_cuda_error(e);
            return TB_ERR_CUDA;
        }
    }
    return TB_OK;
}
