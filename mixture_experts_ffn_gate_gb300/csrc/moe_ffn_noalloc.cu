// moe_ffn_noalloc.cu -- the layer forward pass for callers that cannot
// allocate device memory.
//
// Some callers may not call cudaMalloc (or any allocator) once they are
// running: a serving loop whose latency budget cannot absorb an allocation
// that may synchronise the device or fail under memory pressure at an
// unpredictable moment, or a plugin hosted by an engine that owns all device
// memory through its own pool and forbids other allocations.  This entry
// point gives them the forward pass with its scratch in a fixed, file-scope
// device array instead of a caller- or library-allocated workspace.
//
// The array is MOE_FFN_NOALLOC_SCRATCH_BYTES (16 MiB).  Like every
// __device__ variable it is created in each GPU context that loads the
// library and stays there until the process exits.  All calls share it, so
// two calls whose work overlaps on the GPU (different streams, or different
// host threads without ordering) race on it and give wrong results: order
// them on one stream.  It is the workspace of moe_ffn_forward_ex, so it also
// holds the state that path keeps between calls, under the same rules:
// calls of any shape may follow one another, nothing in it has to start at
// zero, and no one else writes to it.
#include <mutex>

#include "kernels.h"
#include "moe_ffn.h"

namespace {

constexpr size_t kScratchBytes = MOE_FFN_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// Device address of g_noalloc_scratch per device.  In host code the array's
// name only stands in for the symbol; its device address comes from
// cudaGetSymbolAddress, taken once per device with that device current.  The
// address belongs to the context that loaded the library's module, so it is
// looked up again when the current context changes (after cudaDeviceReset
// the module is loaded anew and the array may sit elsewhere, with fresh
// contents).
struct Scratch {
    void *addr = nullptr;
    unsigned long long ctx = 0;
};
Scratch g_scratch[kMaxDevices];
std::mutex g_scratch_mutex;

int scratch_address(void **addr)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    Scratch &sc = g_scratch[dev];
    if (!sc.addr || sc.ctx != moe::current_context_id()) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            sc.addr = nullptr;
            return MOE_ERR_CUDA;
        }
        sc.addr = p;
        sc.ctx = moe::current_context_id();  // the lookup above made the context current if none was
    }
    *addr = sc.addr;
    return MOE_OK;
}

}  // namespace

extern "C" int moe_ffn_forward_noalloc(const void *x_bf16, const float *router_logits_f32,
                                       const void *w_gate_up_bf16, const void *w_down_bf16, int64_t T, int64_t H,
                                       int64_t I, int64_t E, int64_t k, float *out_f32, cudaStream_t stream)
{
    const size_t need = moe_ffn_workspace_bytes(T, H, I, E, k);
    if (need == 0 || T == 0)  // invalid shape or nothing to do: the usual checks answer
        return moe_ffn_forward_ex(x_bf16, router_logits_f32, w_gate_up_bf16, w_down_bf16, T, H, I, E, k, out_f32,
                                  nullptr, 0, nullptr, nullptr, nullptr, stream);
    if (need > kScratchBytes) return MOE_ERR_WORKSPACE_TOO_SMALL;
    void *scratch = nullptr;
    const int st = scratch_address(&scratch);
    if (st != MOE_OK) return st;
    return moe_ffn_forward_ex(x_bf16, router_logits_f32, w_gate_up_bf16, w_down_bf16, T, H, I, E, k, out_f32,
                              scratch, kScratchBytes, nullptr, nullptr, nullptr, stream);
}
