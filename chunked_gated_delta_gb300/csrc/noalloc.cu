// noalloc.cu -- kda_fwd_noalloc: the full forward with its workspace in a
// fixed device array that the library owns, for callers that must not
// allocate device memory themselves.  See include/kda.h for the contract.
#include <mutex>

#include "../../include/kda.h"
#include "internal.h"

namespace {

constexpr size_t kScratchBytes = KDA_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// The scratch array.  Every GPU that loads the library holds one copy until
// the process exits.  In host code `g_kda_scratch` only names the symbol; its
// device address is looked up per device with cudaGetSymbolAddress.
static __device__ __align__(256) uint8_t g_kda_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device (with that device current).  Returns nullptr on failure.
void* scratch_on_current_device(kda_status* err) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        *err = KDA_ERR_CUDA;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_kda_scratch) != cudaSuccess || p == nullptr) {
            *err = KDA_ERR_CUDA;
            return nullptr;
        }
        g_scratch_addr[dev] = p;
    }
    return g_scratch_addr[dev];
}

}  // namespace

extern "C" kda_status kda_fwd_noalloc(const void* q, const void* k, const void* v, const float* g,
                                      const void* beta, float scale, const float* h0,
                                      const int32_t* cu_seqlens, void* o, float* ht,
                                      const kda_dims* dims, void* stream) {
    if (!dims) return KDA_ERR_INVALID_ARG;
    const size_t need = kda_fwd_workspace_size(dims);
    if (need == 0)  // invalid or unsupported dims: let kda_fwd report which, before any launch
        return kda_fwd(q, k, v, g, beta, scale, h0, cu_seqlens, o, ht, dims, nullptr, 0, stream);
    if (need > kScratchBytes) return KDA_ERR_WORKSPACE;
    kda_status err = KDA_OK;
    void* scratch = scratch_on_current_device(&err);
    if (!scratch) return err;
    // every argument of the scan stage is checked before the intra stage
    // enqueues anything (the intra stage checks its own before it launches)
    err = kda::check_scan_args(h0, o, ht, dims, scratch, kScratchBytes);
    if (err != KDA_OK) return err;
    // the two stages in order on the caller's stream, which is kda_fwd's own
    // plan for every problem that fits the scratch (kda_fwd runs chunk ranges
    // on library streams only for workspaces of hundreds of MB)
    kda_status st = kda_fwd_intra(q, k, v, g, beta, cu_seqlens, dims, scratch, kScratchBytes, stream);
    if (st != KDA_OK) return st;
    return kda_fwd_scan(scale, h0, o, ht, dims, scratch, kScratchBytes, stream);
}
