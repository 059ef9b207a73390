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
AttnLaunch plan_attention(const pkv_cache* c, int group, int max_q_len, int num_ctas, int num_sms);
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

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace

using namespace pkv;

extern "C" PKV_API pkv_status pkv_paged_attention_noalloc(
    const pkv_cache* c, const void* q, int32_t num_q_heads, const int32_t* block_tables,
    int32_t max_blocks_per_seq, const int32_t* context_lens, const int32_t* q_lens, int32_t num_seqs,
    int32_t max_q_len, float scale, void* out, int32_t num_ctas, int32_t* device_error, void* stream) {
    // the same argument checks as pkv_paged_attention
    if (!c || !c->k_cache || !c->v_cache || c->num_blocks <= 0 || c->num_kv_heads <= 0) return PKV_ERR_INVALID_ARG;
    if (c->block_size != kBlock || (c->head_dim != 64 && c->head_dim != 128)) return PKV_ERR_UNSUPPORTED;
    if (c->kv_dtype != PKV_KV_BF16 && c->kv_dtype != PKV_KV_FP8_E4M3) return PKV_ERR_UNSUPPORTED;
    if (c->kv_dtype == PKV_KV_FP8_E4M3 && (!c->k_scales || !c->v_scales)) return PKV_ERR_INVALID_ARG;
    if (!aligned16(c->k_cache) || !aligned16(c->v_cache)) return PKV_ERR_INVALID_ARG;
    if (num_seqs < 0 || num_q_heads <= 0 || num_q_heads % c->num_kv_heads) return PKV_ERR_INVALID_ARG;
    if (num_seqs == 0) return PKV_OK;
    if (!q || !out || !block_tables || !context_lens || !q_lens) return PKV_ERR_INVALID_ARG;
    if (max_blocks_per_seq <= 0 || max_q_len < 1 || num_ctas < 0) return PKV_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(out)) return PKV_ERR_INVALID_ARG;
    const int group = num_q_heads / c->num_kv_heads;
    if (max_q_len > 16 || group * max_q_len > 32) return PKV_ERR_UNSUPPORTED;
    if ((int64_t)max_blocks_per_seq * c->num_kv_heads >= (1 << 20)) return PKV_ERR_UNSUPPORTED;   // unit indices stay below 2^20
    if (!(scale == scale)) return PKV_ERR_INVALID_ARG;

    void* scratch = nullptr;
    int sms = 0;
    pkv_status s = device_setup(&scratch, &sms);
    if (s != PKV_OK) return s;
    const AttnLaunch L = plan_attention(c, group, max_q_len, num_ctas, sms);
    const WorkspaceLayout wl = workspace_layout(num_seqs, c->num_kv_heads, c->head_dim, L.rows_pad, L.ncta);
    if (wl.total > (size_t)PKV_NOALLOC_SCRATCH_BYTES) return PKV_ERR_WORKSPACE;   // beyond the fixed maximum

    cudaStream_t st = (cudaStream_t)stream;
    // The error word and the merge tickets must start at zero; the partials need not.
    if (cudaMemsetAsync(scratch, 0, wl.partials_off, st) != cudaSuccess) return PKV_ERR_CUDA;

    AttnParams p;
    p.k_cache = (const uint8_t*)c->k_cache;
    p.v_cache = (const uint8_t*)c->v_cache;
    p.k_scales = c->k_scales;
    p.v_scales = c->v_scales;
    p.q = (const __nv_bfloat16*)q;
    p.out = (__nv_bfloat16*)out;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.q_lens = q_lens;
    p.err = device_error ? (int*)device_error : (int*)scratch;
    p.tickets = (int*)((uint8_t*)scratch + wl.tickets_off);
    p.partials = (float*)((uint8_t*)scratch + wl.partials_off);
    p.num_blocks = c->num_blocks;
    p.num_seqs = num_seqs;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = c->num_kv_heads;
    p.group = group;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.max_q_len = max_q_len;
    p.rows = group * max_q_len;
    p.rows_pad = L.rows_pad;
    p.slot_floats = (int)wl.slot_floats;
    p.scale_log2 = scale * kLog2e;
    p.hg = L.hg;
    const int E = c->kv_dtype == PKV_KV_FP8_E4M3 ? 1 : 2;
    return launch_attention(L, p, c->head_dim, E, st) == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}
