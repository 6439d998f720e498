// rpa_noalloc.cu -- rpa_forward_noalloc: the forward call without any allocation.
//
// Some callers cannot allocate device memory at the point where they run
// attention: code executing under a custom or arena allocator that owns all of
// the device memory, engines that forbid cudaMalloc/cudaFree on the serving path
// because those calls synchronise the device, and hosts that embed the
// library through a plain C interface with no allocator to hand over.  For
// them this entry point runs the same planner, attention and combine kernels
// as rpa_forward, but its workspace (plan, work items and split-KV partials)
// lives in one fixed-size array in the library's own device memory,
// reserved when the library's module is loaded on each GPU and kept until
// the process exits.  Nothing here calls cudaMalloc, cudaFree or any other
// allocating routine.
#include <string.h>

#include <mutex>

#include "rpa_internal.cuh"

using namespace rpa;

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB per GPU
constexpr int kMaxDevices = 64;

// The scratch array itself.  Host code must not take its address directly:
// the symbol's host-side name is only a stand-in for the device object.
static __device__ __align__(256) unsigned char g_rpa_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void* g_scratch_dev[kMaxDevices];
// occupancy per device and kernel choice: [device][D: 64, 128, 256, latent][KvType][8-row decode tiles]
int g_dec_bps[kMaxDevices][4][5][2];
int g_pf_bps[kMaxDevices][4][5][2];
bool g_ready[kMaxDevices][4][5][2];

int d_index(const KernelSet& ks) { return ks.mla ? 3 : ks.D == 64 ? 0 : ks.D == 128 ? 1 : 2; }

// Once per device (and per head size / K/V type for the kernel attributes), with that device
// current: fetch the scratch array's device address and set the kernels' shared-memory limits.
// None of this allocates.  A kernel that cannot be resident is refused here, before anything is
// enqueued (as rpa_create does).
int setup(int dev, KernelSet* ks, void** scratch) {
    if (dev < 0 || dev >= kMaxDevices) return RPA_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_dev[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_rpa_scratch) != cudaSuccess || !ptr) {
            cudaGetLastError();
            return RPA_ERR_CUDA;
        }
        g_scratch_dev[dev] = ptr;
    }
    const int di = d_index(*ks), kt = ks->kt, r8 = ks->dec_rows == 8 ? 1 : 0;
    if (!g_ready[dev][di][kt][r8]) {
        if (kernels_occupancy(ks) != cudaSuccess) {
            cudaGetLastError();
            return RPA_ERR_CUDA;
        }
        g_dec_bps[dev][di][kt][r8] = ks->dec_bps;
        g_pf_bps[dev][di][kt][r8] = ks->pf_bps;
        g_ready[dev][di][kt][r8] = true;
    }
    ks->dec_bps = g_dec_bps[dev][di][kt][r8];
    ks->pf_bps = g_pf_bps[dev][di][kt][r8];
    *scratch = g_scratch_dev[dev];
    return RPA_OK;
}

}  // namespace

extern "C" int rpa_forward_noalloc(const RpaCfg* cfg, const void* q, const void* kv_pages,
                                   const int32_t* kv_lens, const int32_t* page_indices,
                                   const int32_t* cu_q_lens, int32_t num_seqs, void* o, void* stream) {
    const int v = rpa_validate_cfg(cfg);
    if (v != RPA_OK) return v;
    const RpaCfg& c = *cfg;
    if (num_seqs < 0 || num_seqs > c.max_num_seqs) return RPA_ERR_INVALID_ARG;
    if (!kv_pages || !kv_lens || !page_indices || !cu_q_lens) return RPA_ERR_INVALID_ARG;
    if (c.num_q_tokens > 0 && (!q || !o)) return RPA_ERR_INVALID_ARG;
    auto misaligned = [](const void* p, size_t a) { return ((uintptr_t)p % a) != 0; };
    if ((q && misaligned(q, 16)) || (o && misaligned(o, 16)) || misaligned(kv_pages, 16) ||
        misaligned(kv_lens, 4) || misaligned(page_indices, 4) || misaligned(cu_q_lens, 4))
        return RPA_ERR_INVALID_ARG;

    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return RPA_ERR_CUDA;
    }
    KernelSet ks;
    kernels_choose(c, sms, &ks);  // the same kernels and tiles as rpa_create
    void* scratch = nullptr;
    const int su = setup(dev, &ks, &scratch);
    if (su != RPA_OK) return su;
    kernels_capacity(c, &ks);  // the same worst-case workspace as rpa_create's
    if (workspace_bytes(c, ks) > kNoAllocScratchBytes) return RPA_ERR_NO_ALLOC_LIMIT;
    const Workspace ws = workspace_carve(c, ks, scratch);

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // the array keeps the previous call's contents: start the control block at zero
    if (cudaMemsetAsync(ws.ctrl, 0, kCtrlWords * sizeof(int), st) != cudaSuccess) {
        cudaGetLastError();
        return RPA_ERR_CUDA;
    }
    MapCache maps;  // descriptors are encoded on the host stack for this call
    memset(&maps, 0, sizeof maps);
    EnqueueOpts eo;
    memset(&eo, 0, sizeof eo);
    eo.st = st;
    eo.conc = 0;  // one stream: decode and prefill run one after the other on all SMs
    eo.timeout_ns = 1000000000ull;
    return enqueue_forward(c, ks, ws, &maps, q, kv_pages, kv_lens, page_indices, cu_q_lens, num_seqs, o, eo);
}
