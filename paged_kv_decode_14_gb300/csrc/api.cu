// C ABI of libpagedkv: argument checks, grid planning and kernel dispatch.
// Declarations and contracts: include/pagedkv.h.
#include <algorithm>
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "../../include/pagedkv_kvmgr.h"

namespace pkv {
cudaError_t launch_append(const pkv_cache& c, const void* k_new, const void* v_new, const int64_t* slots,
                          int64_t num_tokens, int* err, cudaStream_t st, int num_sms);
cudaError_t launch_append_rope(const pkv_cache& c, const void* k_new, const void* v_new, const int64_t* slots,
                               int64_t T, const int32_t* positions, double theta, void* q, int Hq, bool autoscale,
                               int* err, cudaStream_t st, int num_sms);
cudaError_t launch_copy_blocks(const pkv_cache& c, const int32_t* pairs, int n, float* k_scales, float* v_scales,
                               cudaStream_t st, int num_sms);
cudaError_t launch_attention_simt(const AttnParams& p, int head_dim, int elem_bytes, int ncta, cudaStream_t st);
cudaError_t launch_attention_tc(const AttnParams& p, int head_dim, bool fp8, int ncta, cudaStream_t st);
cudaError_t launch_prefill(const AttnParams& p, int head_dim, int num_sms, cudaStream_t st);
int simt_rows_pad(int rows);
int tc_heads_per_segment(int num_kv_heads, int rows, bool fp8);

// Kernel choice and grid for one attention call, in virtual kv-heads (vheads
// of group vgroup; kv_split of them per cache kv-head): the tensor-core
// kernel for bf16 caches (R = vgroup * max_q_len <= 32 always) and for FP8
// caches with R <= 8, or R <= 16 at head_dim 128 (the split makes it so for
// every window at head_dim 128 and for windows of up to 8 tokens at 64), one
// persistent CTA per SM with all of its ~227 KiB of shared memory; else (FP8,
// head_dim 64, windows of 9-16 tokens) the CUDA-core kernel (4 CTAs per SM).
// rows_pad: partial-slot rows (the tensor-core kernel keeps up to 32 columns
// of several kv-heads per segment).  Virtual kv-heads that share cache pages
// are never grouped in one segment (its pages are copied as one run).
AttnLaunch plan_attention(const pkv_cache* c, int vgroup, int vheads, int kv_split, int max_q_len, int num_ctas,
                          int num_sms) {
    AttnLaunch L;
    const int rows = vgroup * max_q_len;
    const bool fp8 = c->kv_dtype == PKV_KV_FP8_E4M3;
    L.tc = !fp8 ? rows <= 32 : (rows <= 8 || (c->head_dim == 128 && rows <= 16));
    L.ncta = num_ctas > 0 ? num_ctas : (L.tc ? num_sms : 4 * num_sms);
    L.rows_pad = L.tc ? 32 : simt_rows_pad(rows);
    L.hg = (L.tc && kv_split == 1) ? tc_heads_per_segment(vheads, rows, fp8) : 1;
    return L;
}

cudaError_t launch_attention(const AttnLaunch& L, const AttnParams& p, int head_dim, int elem_bytes, cudaStream_t st) {
    return L.tc ? launch_attention_tc(p, head_dim, elem_bytes == 1, L.ncta, st) : launch_attention_simt(p, head_dim, elem_bytes, L.ncta, st);
}

// Debug settings of the timeout path (pkv_debug_set_wait_limit).
namespace {
constexpr uint64_t kDefaultWaitLimitNs = 2000000000ull;   // 2 s
std::atomic<uint64_t> g_wait_limit_ns{0};
std::atomic<const int*> g_hold{nullptr};
}  // namespace

void fill_debug(AttnParams& p) {
    const uint64_t lim = g_wait_limit_ns.load(std::memory_order_relaxed);
    p.wait_limit_ns = lim ? lim : kDefaultWaitLimitNs;
    p.hold = g_hold.load(std::memory_order_relaxed);
}

namespace {

constexpr int kMaxDevices = 64;
int g_num_sms[kMaxDevices] = {0};
std::mutex g_mu;

int num_sms_current() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_num_sms[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        g_num_sms[dev] = n;
    }
    return g_num_sms[dev];
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

pkv_status check_cache(const pkv_cache* c) {
    if (!c || !c->k_cache || !c->v_cache) return PKV_ERR_INVALID_ARG;
    if (c->num_blocks <= 0 || c->num_kv_heads <= 0) return PKV_ERR_INVALID_ARG;
    if (c->block_size != kBlock) return PKV_ERR_UNSUPPORTED;
    if (c->head_dim != 64 && c->head_dim != 128) return PKV_ERR_UNSUPPORTED;
    if (c->kv_dtype != PKV_KV_BF16 && c->kv_dtype != PKV_KV_FP8_E4M3) return PKV_ERR_UNSUPPORTED;
    if (c->kv_dtype == PKV_KV_FP8_E4M3 && (!c->k_scales || !c->v_scales)) return PKV_ERR_INVALID_ARG;
    if (!aligned16(c->k_cache) || !aligned16(c->v_cache)) return PKV_ERR_INVALID_ARG;
    return PKV_OK;
}

// Workspace sizing without a kernel choice covers either kernel: the larger
// default grid and 32 slot rows.
int default_ctas(int num_sms) { return 4 * num_sms; }

}  // namespace

// Argument checks, virtual kv-heads, kernel choice and parameters of one
// attention call, shared by pkv_paged_attention and
// pkv_paged_attention_noalloc.  On PKV_OK with *empty false, *p is complete
// except for its workspace pointers (err, tickets, partials), which follow
// the layout *wl.  *empty: no sequences, nothing to launch.
pkv_status attention_setup(const pkv_cache* cache, const void* q, int num_q_heads, const int32_t* block_tables,
                           int max_blocks_per_seq, const int32_t* context_lens, const int32_t* q_lens, int num_seqs,
                           int max_q_len, float scale, void* out, int num_ctas, int num_sms, AttnParams* p,
                           AttnLaunch* L, WorkspaceLayout* wl, bool* empty, int max_q_limit) {
    *empty = false;
    pkv_status s = check_cache(cache);
    if (s != PKV_OK) return s;
    if (num_seqs < 0 || num_q_heads <= 0 || num_q_heads % cache->num_kv_heads) return PKV_ERR_INVALID_ARG;
    if (num_seqs == 0) {
        *empty = true;
        return PKV_OK;
    }
    if (!q || !out || !block_tables || !context_lens || !q_lens) return PKV_ERR_INVALID_ARG;
    if (max_blocks_per_seq <= 0 || max_q_len < 1 || num_ctas < 0) return PKV_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(out)) return PKV_ERR_INVALID_ARG;
    if (max_q_len > max_q_limit) return PKV_ERR_UNSUPPORTED;
    const int group = num_q_heads / cache->num_kv_heads;
    const int ks = kv_split_for(group, max_q_len,
                                kv_split_limit(cache->kv_dtype == PKV_KV_FP8_E4M3, cache->head_dim, max_q_len));
    const int vgroup = group / ks, vheads = cache->num_kv_heads * ks;
    if ((int64_t)max_blocks_per_seq * vheads >= (1 << 20)) return PKV_ERR_UNSUPPORTED;   // unit indices stay below 2^20
    if (!(scale == scale)) return PKV_ERR_INVALID_ARG;
    if (num_sms <= 0) return PKV_ERR_CUDA;
    *L = plan_attention(cache, vgroup, vheads, ks, max_q_len, num_ctas, num_sms);
    *wl = workspace_layout(num_seqs, vheads, cache->head_dim, L->rows_pad, L->ncta);

    p->k_cache = (const uint8_t*)cache->k_cache;
    p->v_cache = (const uint8_t*)cache->v_cache;
    p->k_scales = cache->k_scales;
    p->v_scales = cache->v_scales;
    p->q = (const __nv_bfloat16*)q;
    p->out = (__nv_bfloat16*)out;
    p->block_tables = block_tables;
    p->context_lens = context_lens;
    p->q_lens = q_lens;
    p->err = nullptr;
    p->tickets = nullptr;
    p->partials = nullptr;
    p->num_blocks = cache->num_blocks;
    p->num_seqs = num_seqs;
    p->num_q_heads = num_q_heads;
    p->num_kv_heads = vheads;
    p->group = vgroup;
    p->max_blocks_per_seq = max_blocks_per_seq;
    p->max_q_len = max_q_len;
    p->rows = vgroup * max_q_len;
    p->rows_pad = L->rows_pad;
    p->slot_floats = (int)wl->slot_floats;
    p->scale_log2 = scale * kLog2e;
    p->hg = L->hg;
    p->kv_split = ks;
    p->cache_kv_heads = cache->num_kv_heads;
    p->cascade = 0;
    p->group_starts = nullptr;
    p->group_prefix_lens = nullptr;
    p->num_groups = 0;
    p->num_seqs_total = num_seqs;
    p->state_o = nullptr;
    p->state_lse = nullptr;
    fill_debug(*p);
    return PKV_OK;
}

}  // namespace pkv

using namespace pkv;

extern "C" {

PKV_API const char* pkv_version(void) { return "pagedkv 0.1 (sm_103a)"; }

PKV_API const char* pkv_status_string(pkv_status s) {
    switch (s) {
        case PKV_OK: return "ok";
        case PKV_ERR_INVALID_ARG: return "invalid argument";
        case PKV_ERR_UNSUPPORTED: return "unsupported configuration";
        case PKV_ERR_WORKSPACE: return "workspace missing or too small";
        case PKV_ERR_CUDA: return "CUDA error";
        case PKV_ERR_DEVICE_INDEX: return "device-side index, length or value-range error";
        case PKV_ERR_TIMEOUT: return "device-side wait timed out";
        case PKV_ERR_NO_BLOCKS: return "no free cache block and none evictable";
        case PKV_ERR_UNKNOWN_SEQ: return "unknown (or already registered) sequence id";
    }
    return "unknown status";
}

PKV_API pkv_status pkv_paged_kv_append(const pkv_cache* cache, const void* k_new, const void* v_new,
                                       const int64_t* slot_mapping, int64_t num_tokens, int32_t* device_error,
                                       void* stream) {
    pkv_status s = check_cache(cache);
    if (s != PKV_OK) return s;
    if (num_tokens < 0) return PKV_ERR_INVALID_ARG;
    if (num_tokens == 0) return PKV_OK;
    if (!k_new || !v_new || !slot_mapping) return PKV_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new)) return PKV_ERR_INVALID_ARG;
    const int sms = num_sms_current();
    if (sms <= 0) return PKV_ERR_CUDA;
    cudaError_t e = launch_append(*cache, k_new, v_new, slot_mapping, num_tokens, device_error,
                                  (cudaStream_t)stream, sms);
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

PKV_API pkv_status pkv_paged_kv_append_rope(const pkv_cache* cache, const void* k_new, const void* v_new,
                                            const int64_t* slot_mapping, int64_t num_tokens, const int32_t* positions,
                                            float rope_theta, void* q, int32_t num_q_heads,
                                            int32_t fp8_scales_from_values, int32_t* device_error, void* stream) {
    pkv_status s = check_cache(cache);
    if (s != PKV_OK) return s;
    if (num_tokens < 0 || num_tokens > 0x7fffffff) return PKV_ERR_INVALID_ARG;
    if (num_tokens == 0) return PKV_OK;
    if (!k_new || !v_new || !slot_mapping) return PKV_ERR_INVALID_ARG;
    if (positions && !(rope_theta > 0.f)) return PKV_ERR_INVALID_ARG;
    if (q && (!positions || num_q_heads <= 0 || num_q_heads % cache->num_kv_heads)) return PKV_ERR_INVALID_ARG;
    if (fp8_scales_from_values && cache->kv_dtype != PKV_KV_FP8_E4M3) return PKV_ERR_INVALID_ARG;
    if (cache->num_kv_heads > 32) return PKV_ERR_UNSUPPORTED;
    const int sms = num_sms_current();
    if (sms <= 0) return PKV_ERR_CUDA;
    return launch_append_rope(*cache, k_new, v_new, slot_mapping, num_tokens, positions, (double)rope_theta, q,
                              q ? num_q_heads : 0, fp8_scales_from_values != 0, device_error, (cudaStream_t)stream,
                              sms) == cudaSuccess
               ? PKV_OK
               : PKV_ERR_CUDA;
}

PKV_API pkv_status pkv_copy_blocks(const pkv_cache* cache, const int32_t* pairs, int32_t n, float* k_scales,
                                   float* v_scales, void* stream) {
    pkv_status s = check_cache(cache);
    if (s != PKV_OK) return s;
    if (n < 0) return PKV_ERR_INVALID_ARG;
    if (n == 0) return PKV_OK;
    if (!pairs) return PKV_ERR_INVALID_ARG;
    const int sms = num_sms_current();
    if (sms <= 0) return PKV_ERR_CUDA;
    return launch_copy_blocks(*cache, pairs, n, k_scales, v_scales, (cudaStream_t)stream, sms) == cudaSuccess
               ? PKV_OK
               : PKV_ERR_CUDA;
}

PKV_API size_t pkv_attention_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                            int32_t head_dim, int32_t max_q_len, int32_t num_ctas) {
    if (num_seqs < 0 || num_kv_heads <= 0 || num_q_heads <= 0 || num_q_heads % num_kv_heads) return 0;
    if (head_dim <= 0 || max_q_len < 1) return 0;
    if (num_ctas <= 0) num_ctas = default_ctas(num_sms_current());
    if (num_ctas <= 0) return 0;
    // (the cache's dtype is not an argument: the larger of the bf16 and FP8 plans)
    const int group = num_q_heads / num_kv_heads;
    size_t need = 0;
    for (int fp8 = 0; fp8 < 2; ++fp8) {
        const int ks = kv_split_for(group, max_q_len, kv_split_limit(fp8 != 0, head_dim, max_q_len));
        const int rows_pad = max(32, simt_rows_pad((group / ks) * max_q_len));
        need = std::max(need, workspace_layout(num_seqs, num_kv_heads * ks, head_dim, rows_pad, num_ctas).total);
    }
    return need;
}

PKV_API pkv_status pkv_workspace_init(void* workspace, size_t workspace_bytes, void* stream) {
    if (!workspace || workspace_bytes < 256) return PKV_ERR_INVALID_ARG;
    return cudaMemsetAsync(workspace, 0, workspace_bytes, (cudaStream_t)stream) == cudaSuccess ? PKV_OK
                                                                                              : PKV_ERR_CUDA;
}

PKV_API pkv_status pkv_paged_attention(const pkv_cache* cache, const void* q, int32_t num_q_heads,
                                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                                       const int32_t* context_lens, const int32_t* q_lens, int32_t num_seqs,
                                       int32_t max_q_len, float scale, void* out, void* workspace,
                                       size_t workspace_bytes, int32_t num_ctas, void* stream) {
    AttnParams p;
    AttnLaunch L;
    WorkspaceLayout wl;
    bool empty = false;
    const pkv_status s = attention_setup(cache, q, num_q_heads, block_tables, max_blocks_per_seq, context_lens, q_lens,
                                         num_seqs, max_q_len, scale, out, num_ctas, num_sms_current(), &p, &L, &wl,
                                         &empty, 16);
    if (s != PKV_OK || empty) return s;
    if (!workspace) return PKV_ERR_INVALID_ARG;
    if (!aligned16(workspace)) return PKV_ERR_INVALID_ARG;
    if (workspace_bytes < wl.total) return PKV_ERR_WORKSPACE;
    p.err = (int*)workspace;
    p.tickets = (int*)((uint8_t*)workspace + wl.tickets_off);
    p.partials = (float*)((uint8_t*)workspace + wl.partials_off);
    const int E = cache->kv_dtype == PKV_KV_FP8_E4M3 ? 1 : 2;
    cudaError_t e = launch_attention(L, p, cache->head_dim, E, (cudaStream_t)stream);
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

PKV_API pkv_status pkv_paged_prefill(const pkv_cache* cache, const void* q, int32_t num_q_heads,
                                     const int32_t* block_tables, int32_t max_blocks_per_seq,
                                     const int32_t* context_lens, const int32_t* q_lens, int32_t num_seqs,
                                     int32_t max_q_len, float scale, void* out, int32_t* device_error,
                                     void* stream) {
    pkv_status s = check_cache(cache);
    if (s != PKV_OK) return s;
    if (num_seqs < 0 || num_q_heads <= 0 || num_q_heads % cache->num_kv_heads) return PKV_ERR_INVALID_ARG;
    if (cache->kv_dtype != PKV_KV_BF16) return PKV_ERR_UNSUPPORTED;
    const int group = num_q_heads / cache->num_kv_heads;
    if (128 % group) return PKV_ERR_UNSUPPORTED;
    if (num_seqs == 0) return PKV_OK;
    if (!q || !out || !block_tables || !context_lens || !q_lens) return PKV_ERR_INVALID_ARG;
    if (max_blocks_per_seq <= 0 || max_q_len < 1) return PKV_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(out)) return PKV_ERR_INVALID_ARG;
    if (!(scale == scale)) return PKV_ERR_INVALID_ARG;
    const int64_t qblocks = ((int64_t)max_q_len * group + 255) / 256;
    if ((int64_t)num_seqs * cache->num_kv_heads * qblocks > 0x7fffffff) return PKV_ERR_UNSUPPORTED;
    AttnParams p = {};
    p.k_cache = (const uint8_t*)cache->k_cache;
    p.v_cache = (const uint8_t*)cache->v_cache;
    p.q = (const __nv_bfloat16*)q;
    p.out = (__nv_bfloat16*)out;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.q_lens = q_lens;
    p.err = device_error;
    p.num_blocks = cache->num_blocks;
    p.num_seqs = num_seqs;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = cache->num_kv_heads;
    p.group = group;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.max_q_len = max_q_len;
    p.scale_log2 = scale * kLog2e;
    p.hg = 1;
    p.kv_split = 1;
    p.cache_kv_heads = cache->num_kv_heads;
    p.num_seqs_total = num_seqs;
    fill_debug(p);
    const int sms = num_sms_current();
    if (sms <= 0) return PKV_ERR_CUDA;
    return launch_prefill(p, cache->head_dim, sms, (cudaStream_t)stream) == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

PKV_API void pkv_debug_set_wait_limit(uint64_t limit_ns, const int32_t* hold_flag) {
    g_wait_limit_ns.store(limit_ns, std::memory_order_relaxed);
    g_hold.store(hold_flag, std::memory_order_relaxed);
}

// Workspace of a cascade call: the prefix pass's (groups as sequences), the
// suffix pass's, then the prefix states (fp32 output rows and their
// log2-sum-exp), each 256-byte aligned.
struct CascadeLayout {
    size_t a_off, b_off, o_off, lse_off, total;
};
static CascadeLayout cascade_layout(size_t a_bytes, size_t b_bytes, int64_t rows, int Hq, int D) {
    CascadeLayout c;
    c.a_off = 0;
    c.b_off = align_up(a_bytes, 256);
    c.o_off = align_up(c.b_off + b_bytes, 256);
    c.lse_off = align_up(c.o_off + (size_t)rows * Hq * D * 4, 256);
    c.total = align_up(c.lse_off + (size_t)rows * Hq * 4, 256);
    return c;
}

PKV_API size_t pkv_cascade_workspace_size(int32_t num_seqs, int32_t num_groups, int32_t num_q_heads,
                                          int32_t num_kv_heads, int32_t head_dim, int32_t max_q_len,
                                          int32_t max_group_q_len) {
    if (num_groups < 0 || max_group_q_len < 1 || max_q_len < 1) return 0;
    const size_t a = pkv_attention_workspace_size(num_groups, num_q_heads, num_kv_heads, head_dim, max_group_q_len, 0);
    const size_t b = pkv_attention_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, max_q_len, 0);
    if (!a || !b) return 0;
    return cascade_layout(a, b, (int64_t)num_seqs * max_q_len, num_q_heads, head_dim).total;
}

PKV_API pkv_status pkv_paged_attention_cascade(const pkv_cache* cache, const void* q, int32_t num_q_heads,
                                               const int32_t* block_tables, int32_t max_blocks_per_seq,
                                               const int32_t* context_lens, const int32_t* q_lens, int32_t num_seqs,
                                               int32_t max_q_len, const int32_t* group_starts,
                                               const int32_t* group_prefix_lens, int32_t num_groups,
                                               int32_t max_group_q_len, float scale, void* out, void* workspace,
                                               size_t workspace_bytes, void* stream) {
    if (num_groups < 1 || !group_starts || !group_prefix_lens || max_group_q_len < 1) return PKV_ERR_INVALID_ARG;
    if (!workspace || !aligned16(workspace)) return PKV_ERR_INVALID_ARG;
    const int sms = num_sms_current();
    AttnParams pa, pb;
    AttnLaunch la, lb;
    WorkspaceLayout wa, wb;
    bool empty = false;
    // the prefix pass: groups as sequences, their whole q windows (up to 32 rows), prefix lengths as contexts
    pkv_status s = attention_setup(cache, q, num_q_heads, block_tables, max_blocks_per_seq, group_prefix_lens, q_lens,
                                   num_groups, max_group_q_len, scale, out, 0, sms, &pa, &la, &wa, &empty, 32);
    if (s != PKV_OK) return s;
    s = attention_setup(cache, q, num_q_heads, block_tables, max_blocks_per_seq, context_lens, q_lens, num_seqs,
                        max_q_len, scale, out, 0, sms, &pb, &lb, &wb, &empty, 16);
    if (s != PKV_OK || empty) return s;
    if (!la.tc || !lb.tc || cache->kv_dtype != PKV_KV_BF16) return PKV_ERR_UNSUPPORTED;   // bf16, tensor-core passes
    const CascadeLayout cl = cascade_layout(wa.total, wb.total, (int64_t)num_seqs * max_q_len, num_q_heads,
                                            cache->head_dim);
    if (workspace_bytes < cl.total) return PKV_ERR_WORKSPACE;
    uint8_t* w = (uint8_t*)workspace;
    float* so = (float*)(w + cl.o_off);
    float* sl = (float*)(w + cl.lse_off);
    pa.err = (int*)(w + cl.a_off);
    pa.tickets = (int*)(w + cl.a_off + wa.tickets_off);
    pa.partials = (float*)(w + cl.a_off + wa.partials_off);
    pa.cascade = 1;
    pa.group_starts = group_starts;
    pa.num_groups = num_groups;
    pa.num_seqs_total = num_seqs;
    pa.state_o = so;
    pa.state_lse = sl;
    pb.err = (int*)(w + cl.a_off);                             // one error word for both passes
    pb.tickets = (int*)(w + cl.b_off + wb.tickets_off);
    pb.partials = (float*)(w + cl.b_off + wb.partials_off);
    pb.cascade = 2;
    pb.group_starts = group_starts;
    pb.group_prefix_lens = group_prefix_lens;
    pb.num_groups = num_groups;
    pb.state_o = so;
    pb.state_lse = sl;
    const int E = cache->kv_dtype == PKV_KV_FP8_E4M3 ? 1 : 2;
    cudaError_t e = launch_attention(la, pa, cache->head_dim, E, (cudaStream_t)stream);
    if (e == cudaSuccess) e = launch_attention(lb, pb, cache->head_dim, E, (cudaStream_t)stream);
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

PKV_API pkv_status pkv_read_device_error(void* error_word, int32_t* code, void* stream) {
    if (!error_word || !code) return PKV_ERR_INVALID_ARG;
    int32_t h = 0;
    cudaStream_t st = (cudaStream_t)stream;
    if (cudaMemcpyAsync(&h, error_word, sizeof(h), cudaMemcpyDeviceToHost, st) != cudaSuccess) return PKV_ERR_CUDA;
    if (cudaMemsetAsync(error_word, 0, sizeof(h), st) != cudaSuccess) return PKV_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return PKV_ERR_CUDA;
    *code = h;
    if (h == 0) return PKV_OK;
    return (h & PKV_DEVERR_TIMEOUT) ? PKV_ERR_TIMEOUT : PKV_ERR_DEVICE_INDEX;
}

}  // extern "C"
