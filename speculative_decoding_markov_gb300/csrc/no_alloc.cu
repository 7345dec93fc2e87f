// no_alloc.cu - greedy verification for callers that cannot allocate.
//
// sdm_verify needs a scratch buffer for its per-chunk argmax partials, and the
// caller normally provides it (sized by sdm_workspace_size).  Some callers
// cannot: an inference server that reserves all device memory at start-up and
// hands out no more, a host framework whose own caching allocator must account
// for every byte (a library calling cudaMalloc behind its back breaks that),
// or a latency-critical loop where the implicit device synchronisation of
// cudaMalloc / cudaFree is not acceptable.  sdm_verify_greedy_static serves
// them: its scratch is a fixed array in device memory that belongs to this
// library.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds kStaticScratchBytes of it until the process exits.  Host code
// cannot use the array's name as a device address: the address is looked up
// with cudaGetSymbolAddress once per device, with that device current, on the
// first call made on that device.  The lookup is kept together with the CUDA
// context it was made in; a call made in another context (the device was
// reset, or its primary context released and created again, which loads the
// module again and may move the array) looks it up again.
#include <cudaTypedefs.h>

#include <mutex>

#include "internal.h"

namespace {

constexpr size_t kStaticScratchBytes = 1u << 20;                       // 1 MiB
constexpr size_t kStaticKeys = kStaticScratchBytes / sizeof(unsigned long long);
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned long long g_verify_scratch[kStaticKeys];

std::mutex g_setup_mutex;
unsigned long long* g_scratch_ptr[kMaxDevices] = {};
CUcontext g_scratch_ctx[kMaxDevices] = {};

// cuCtxGetCurrent through the runtime's driver entry point (the library does
// not link the driver library itself).
CUresult current_context(CUcontext* ctx) {
    static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !p)
            return CUDA_ERROR_NOT_FOUND;
        fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    }
    return fn(ctx);
}

// Device address of the scratch array for the current device and context
// (set-up on the first call per device, again after a context change).
// Returns nullptr on failure.
unsigned long long* scratch_for_current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    // NULL until the runtime has made a context current on this thread
    CUcontext ctx = nullptr;
    if (current_context(&ctx) != CUDA_SUCCESS) return nullptr;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_ptr[dev] || !ctx || g_scratch_ctx[dev] != ctx) {
        // the lookup makes the device's primary context current if it is not
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_verify_scratch) != cudaSuccess || !p) return nullptr;
        if (current_context(&ctx) != CUDA_SUCCESS || !ctx) return nullptr;
        g_scratch_ptr[dev] = static_cast<unsigned long long*>(p);
        g_scratch_ctx[dev] = ctx;
    }
    return g_scratch_ptr[dev];
}

}  // namespace

extern "C" sdm_status sdm_verify_greedy_static(sdm_vmode mode, const void* target, sdm_dtype dtT, int row_capacity,
                                               const int32_t* cu_seqlens, const int32_t* draft,
                                               const int32_t* budget, int R, int gamma, int V, int32_t* accept,
                                               int32_t* ceiling, int32_t* out_tok, int32_t* n_out,
                                               int32_t* dev_status, void* stream) {
    using namespace sdm;
    if (!target || !cu_seqlens || !draft || !accept || !out_tok || !n_out) return SDM_ERR_INVALID_ARG;
    if (R <= 0 || gamma <= 0 || V <= 0 || row_capacity <= 0) return SDM_ERR_INVALID_ARG;
    if (mode != SDM_STATIC && mode != SDM_COMPACT && mode != SDM_CAP_ACCEPT) return SDM_ERR_INVALID_ARG;
    if (dtT != SDM_BF16 && dtT != SDM_FP32) return SDM_ERR_INVALID_ARG;
    if (mode == SDM_CAP_ACCEPT && !budget) return SDM_ERR_INVALID_ARG;
    if (V < 8 || V % 8 != 0 || (reinterpret_cast<uintptr_t>(target) & 15u) != 0) return SDM_ERR_UNSUPPORTED;
    const int fp32 = dtT == SDM_FP32;
    const int chunk = fp32 ? kChunkFp32 : kChunkBf16;   // the streaming work items of sdm_verify
    const int n_chunks = n_chunks_of(V, fp32);
    // one partial key per (row, chunk) must fit the fixed array
    if (static_cast<size_t>(row_capacity) * static_cast<size_t>(n_chunks) > kStaticKeys) return SDM_ERR_WORKSPACE;
    unsigned long long* keys = scratch_for_current_device();
    if (!keys) return SDM_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    StreamParams sp = {};
    sp.base = target;
    sp.fp32 = fp32;
    sp.V = V;
    sp.chunk = chunk;
    sp.n_chunks = n_chunks;
    sp.count = cu_seqlens + R;
    sp.n_items = row_capacity;
    sp.inv_t = 1.0f;
    sp.keys = keys;   // every (row, chunk) partial read below is written first in this call (rows below cu[R])
    if (launch_stream(STREAM_ARGMAX, sp, row_capacity, s) != cudaSuccess) return SDM_ERR_CUDA;
    if (launch_verify_greedy_finalize(mode, cu_seqlens, draft, budget, keys, n_chunks, R, gamma, V, row_capacity,
                                      accept, ceiling, out_tok, n_out, dev_status, s) != cudaSuccess)
        return SDM_ERR_CUDA;
    return SDM_OK;
}
