// pkv_paged_attention_noalloc: paged attention for callers that cannot
// allocate device memory.
//
// Who needs it: a caller that owns no device allocator of its own -- for
// example a plugin or foreign-language host that can only hand over the
// tensors it already holds, or a serving loop whose device memory budget is
// fixed at start-up and must not grow or fragment on the decode path.  Such a
// caller cannot provide the attention workspace (the split partials, the merge
// tickets and the error word).  This entry point keeps that scratch in a
// file-scope device array instead, so the caller passes only inputs and
// outputs.  The pages have no counterpart of this entry point.
//
// The array, PKV_NOALLOC_SCRATCH_BYTES (32 MiB), is part of the library's
// device image: every GPU that loads libpagedkv.so holds it until the process
// exits.  All calls share it and it keeps the last call's contents, so calls
// whose kernels overlap on the GPU (different streams, or different host
// threads on one device) race and must be serialised by the caller.
#include <mutex>

#include "common.cuh"

namespace pkv {
pkv_status attention_setup(const pkv_cache* cache, const void* q, int num_q_heads, const int32_t* block_tables,
                           int max_blocks_per_seq, const int32_t* context_lens, const int32_t* q_lens, int num_seqs,
                           int max_q_len, float scale, void* out, int num_ctas, int num_sms, AttnParams* p,
                           AttnLaunch* L, WorkspaceLayout* wl, bool* empty, int max_q_limit);
cudaError_t launch_attention(const AttnLaunch& L, const AttnParams& p, int head_dim, int elem_bytes, cudaStream_t st);
}  // namespace pkv

static __device__ __align__(256) uint8_t g_pkv_noalloc_scratch[PKV_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {nullptr};
int g_num_sms[kMaxDevices] = {0};
std::mutex g_mu;

// Device address of the scratch array and the SM count of the current
// device.  The first call on a device looks both up (with that device
// current) and caches them.
pkv_status device_setup(void** scratch, int* sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PKV_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_pkv_noalloc_scratch) != cudaSuccess || p == nullptr) return PKV_ERR_CUDA;
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            return PKV_ERR_CUDA;
        g_scratch_addr[dev] = p;
        g_num_sms[dev] = n;
    }
    *scratch = g_scratch_addr[dev];
    *sms = g_num_sms[dev];
    return PKV_OK;
}

}  // namespace

using namespace pkv;

extern "C" PKV_API pkv_status pkv_paged_attention_noalloc(
    const pkv_cache* c, const void* q, int32_t num_q_heads, const int32_t* block_tables,
    int32_t max_blocks_per_seq, const int32_t* context_lens, const int32_t* q_lens, int32_t num_seqs,
    int32_t max_q_len, float scale, void* out, int32_t num_ctas, int32_t* device_error, void* stream) {
    // the same argument checks and parameters as pkv_paged_attention
    void* scratch = nullptr;
    int sms = 0;
    AttnParams p;
    AttnLaunch L;
    WorkspaceLayout wl;
    bool empty = false;
    pkv_status s = device_setup(&scratch, &sms);
    if (s != PKV_OK) return s;
    s = pkv::attention_setup(c, q, num_q_heads, block_tables, max_blocks_per_seq, context_lens, q_lens, num_seqs,
                             max_q_len, scale, out, num_ctas, sms, &p, &L, &wl, &empty, 16);
    if (s != PKV_OK || empty) return s;
    if (wl.total > (size_t)PKV_NOALLOC_SCRATCH_BYTES) return PKV_ERR_WORKSPACE;   // beyond the fixed maximum

    cudaStream_t st = (cudaStream_t)stream;
    // The error word and the merge tickets must start at zero; the partials need not.
    if (cudaMemsetAsync(scratch, 0, wl.partials_off, st) != cudaSuccess) return PKV_ERR_CUDA;
    p.err = device_error ? (int*)device_error : (int*)scratch;
    p.tickets = (int*)((uint8_t*)scratch + wl.tickets_off);
    p.partials = (float*)((uint8_t*)scratch + wl.partials_off);
    const int E = c->kv_dtype == PKV_KV_FP8_E4M3 ? 1 : 2;
    return launch_attention(L, p, c->head_dim, E, st) == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}
