// tb_noalloc.cu -- PatchGroupNorm without any device allocation.
//
// For callers that cannot allocate device memory (a host framework that owns
// every allocation through its own pool, or a latency-critical path where
// cudaMalloc is not allowed): the per-patch partial statistics that
// tb_patch_gn_stats writes and tb_patch_gn_apply reads live in a fixed array
// compiled into this library rather than in a caller-provided buffer.  The
// kernels and their arguments are otherwise the existing ones.
//
// The array holds TB_NOALLOC_MAX_PARTIALS 16-byte records (1 MiB) on every
// device that loads the library, for the life of the process: the
// TB_GN_PARTS records of each of up to 8192 (patch, sample, group) units.
// Calls share it: each call's statistics kernel writes every record its
// apply kernel reads, so nothing needs clearing between calls, but calls
// whose work overlaps on the GPU race on it.
#include <mutex>

#include "tb_internal.h"
#include "tileblend.h"

#define TB_API extern "C" __attribute__((visibility("default")))

namespace {

static __device__ __align__(256) tb::GnPartial g_noalloc_partials[TB_NOALLOC_MAX_PARTIALS];

constexpr int MAX_DEVICES = 64;

// The scratch array's device address, as looked up in one CUDA context.  A
// device reset destroys the context and the library's module with it; the
// module loaded into the next context may place the array elsewhere.  So
// the cached address is tied to the process-unique id of the context it was
// looked up in, and a call in any other context looks it up again.
struct ScratchAddr {
    unsigned long long ctx_id;
    void* addr;
};
std::mutex g_addr_mu;
ScratchAddr g_addr[MAX_DEVICES] = {};

// Device address of the scratch array in the current context.  Host code
// sees the array's name only as a host-side stand-in, so the address comes
// from cudaGetSymbolAddress, looked up once per device (and again after the
// device's context has been replaced), with that device current.
tb_status scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        tb::record_cuda_error(e);
        return TB_ERR_CUDA;
    }
    if (dev < 0 || dev >= MAX_DEVICES) return TB_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_addr_mu);
    const unsigned long long id = tb::current_context_id();
    ScratchAddr& c = g_addr[dev];
    if (c.addr == nullptr || id == 0 || id != c.ctx_id) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_partials);
        if (e != cudaSuccess || p == nullptr) {
            tb::record_cuda_error(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
            return TB_ERR_CUDA;
        }
        c.addr = p;
        c.ctx_id = tb::current_context_id();  // bound now, if it was not before
    }
    *out = c.addr;
    return TB_OK;
}

}  // namespace

TB_API tb_status tb_patch_group_norm_noalloc(const void* const* patches, void* const* outs, int32_t P, tb_dtype dtype,
                                             int64_t N, int64_t C, const int64_t* spatial, int32_t G,
                                             const void* gamma, const void* beta, float eps, int32_t silu,
                                             void* stream) {
    if (P < 1 || N < 0 || C < 0 || G < 1) return TB_ERR_SHAPE;
    if ((double)P * (double)N * (double)G * TB_GN_PARTS > (double)TB_NOALLOC_MAX_PARTIALS) return TB_ERR_UNSUPPORTED;
    // checks the apply step would make, done before the statistics launch
    if (!(eps >= 0.0f) || eps > 3.0e38f) return TB_ERR_SHAPE;
    if (outs == nullptr) return TB_ERR_NULL;
    if (N == 0 || C == 0) {
        return tb_patch_gn_apply(patches, outs, P, dtype, N, C, spatial, G, nullptr, gamma, beta, eps, silu, stream);
    }
    if (spatial != nullptr)
        for (int p = 0; p < P; ++p)
            if (spatial[p] > 0 && outs[p] == nullptr) return TB_ERR_NULL;
    void* scratch = nullptr;
    tb_status st = scratch_address(&scratch);
    if (st != TB_OK) return st;
    st = tb_patch_gn_stats(patches, P, dtype, N, C, spatial, G, reinterpret_cast<tb_gn_partial*>(scratch), stream);
    if (st != TB_OK) return st;
    return tb_patch_gn_apply(patches, outs, P, dtype, N, C, spatial, G, reinterpret_cast<const tb_gn_partial*>(scratch),
                             gamma, beta, eps, silu, stream);
}
