// pkv_noalloc.cu -- paged decode for callers that cannot allocate device memory.
//
// pkv_paged_decode needs a caller-owned workspace for its split-K partials.
// Some callers cannot make one: code that runs while another component holds
// a stream capture open in global mode (cudaMalloc is not allowed then), a
// plugin inside an engine whose allocator owns all device memory and forbids
// direct cudaMalloc, or a latency-bound loop that cannot afford cudaMalloc's
// implicit device synchronisation.  pkv_paged_decode_noalloc gives them the
// same decode with the partials in a fixed, library-owned device array.
//
// The array is a file-scope __device__ object of kStaticScratchBytes (8 MiB):
// every GPU that loads the library holds it until the process exits.  Host
// code cannot use the array's name as a device address, so the first call on
// each device looks the address up with cudaGetSymbolAddress (with that
// device current) and caches it.  Nothing here calls cudaMalloc or cudaFree.
#include <mutex>

#include "pkv.h"
#include "pkv_launch.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(8) << 20;
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
void *g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of g_static_scratch on the current device (set up once).
int scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PKV_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess) return PKV_ERR_CUDA;
        g_scratch_addr[dev] = ptr;
    }
    *out = g_scratch_addr[dev];
    return PKV_OK;
}

}  // namespace

extern "C" {

int pkv_paged_decode_noalloc(const pkv_kvcache *c, int32_t layer_id, const void *q, void *o,
                             int32_t n_heads, float sm_scale, void *stream) {
    if (!c || n_heads <= 0 || c->head_dim <= 0) return PKV_ERR_ARG;
    if (c->batch <= 0) return pkv_paged_decode(c, layer_id, q, o, n_heads, sm_scale, nullptr, stream);
    // As many splits per (entry, head) as the fixed array holds, at most the
    // decode kernel's own limit.
    int32_t splits = 0;
    for (int32_t s = 1; s <= pkv::kDecodeMaxSplits; ++s) {
        const size_t need = pkv_workspace_bytes(c->batch, n_heads, c->head_dim, s);
        if (need == 0 || need > kStaticScratchBytes) break;
        splits = s;
    }
    if (splits == 0) {
        // Not even one split per (entry, head) fits.  Contexts that one split
        // covers need no partials: the decode writes o directly.
        if (c->max_len <= pkv::kDecodeMaxChunk)
            return pkv_paged_decode(c, layer_id, q, o, n_heads, sm_scale, nullptr, stream);
        return PKV_ERR_WORKSPACE;
    }
    void *base = nullptr;
    int rc = scratch_address(&base);
    if (rc) return rc;
    pkv_workspace ws;
    rc = pkv_workspace_init(base, kStaticScratchBytes, c->batch, n_heads, c->head_dim, splits, &ws);
    if (rc) return rc;
    return pkv_paged_decode(c, layer_id, q, o, n_heads, sm_scale, &ws, stream);
}

}  // extern "C"
