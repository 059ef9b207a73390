// paged_kv_append: write one step's new K/V rows into their cache slots
// (lfm25-inference file list: kernels/kv_cache.cu, scheduler/slots.rs).
//
// One thread per (token, kv-head, 16-byte cache chunk, K|V).  For a bf16
// cache the chunk is 8 bf16 values copied as one 16-byte store; for an FP8
// cache it is 16 values, each divided by its (block, kv-head) scale in IEEE
// fp32 (round to nearest) and converted by CUDA's E4M3 conversion with
// round-to-nearest-even and saturation to +-448.
#include "common.cuh"

namespace pkv {

// At most 32 registers a thread (bf16), so that a 32-thread CTA fits beside a resident
// attention CTA (384 threads x 168 registers leave 1024 of an SM's 65536): a
// decode step's append is then already waiting on the SMs when the attention
// before it ends.
template <int E>
__global__ void __maxnreg__(E == 2 ? 32 : 48) append_kernel(const uint8_t* __restrict__ k_new, const uint8_t* __restrict__ v_new,
                                                     const int64_t* __restrict__ slots, int64_t num_tokens, int Hkv,
                                                     int D, int64_t num_blocks, uint8_t* k_cache, uint8_t* v_cache,
                                                     const float* __restrict__ k_scales,
                                                     const float* __restrict__ v_scales, int* err) {
    griddep_launch();                            // the attention that follows may start its set-up
    const int NCH = D * E / 16;                  // 16-byte chunks per token row in the cache
    const int64_t per_tok = (int64_t)Hkv * NCH * 2;
    const int64_t total = num_tokens * per_tok;
    const int64_t idx0 = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    // The thread's first chunk (a decode step's only one): its slot and source are read before
    // the dependency wait (the previous kernel -- the last step's attention -- does not write
    // them), so that only the stores follow the wait.  Scales are read after it.
    int64_t s0 = -1;
    uint4 a0 = make_uint4(0, 0, 0, 0), b0 = a0;
    if (idx0 < total) {
        const int64_t t = idx0 / per_tok;
        int rem = (int)(idx0 % per_tok);
        const int which = rem & 1;
        rem >>= 1;
        const int g = rem / NCH, ch = rem % NCH;
        s0 = slots[t];
        const uint8_t* src = (which ? v_new : k_new) + (((size_t)t * Hkv + g) * D) * 2;
        if constexpr (E == 2) {
            a0 = __ldg(reinterpret_cast<const uint4*>(src + ch * 16));
        } else {
            a0 = __ldg(reinterpret_cast<const uint4*>(src + ch * 32));
            b0 = __ldg(reinterpret_cast<const uint4*>(src + ch * 32 + 16));
        }
    }
    griddep_wait();                              // the previous kernel's reads and writes are done
    for (int64_t idx = idx0; idx < total; idx += (int64_t)gridDim.x * blockDim.x) {
        const bool first = idx == idx0;
        const int64_t t = idx / per_tok;
        int rem = (int)(idx % per_tok);
        const int which = rem & 1;               // 0 = K, 1 = V
        rem >>= 1;
        const int g = rem / NCH, ch = rem % NCH;
        const int64_t s = first ? s0 : slots[t];
        if (s < 0) continue;
        const int64_t blk = s / kBlock;
        const int off = (int)(s % kBlock);
        if (blk >= num_blocks) {
            if (which == 0 && g == 0 && ch == 0) raise_error(err, PKV_DEVERR_SLOT);
            continue;
        }
        const uint8_t* src = (which ? v_new : k_new) + (((size_t)t * Hkv + g) * D) * 2;
        uint8_t* page = (which ? v_cache : k_cache) + ((size_t)blk * Hkv + g) * (size_t)(kBlock * D * E);
        uint4* dst = reinterpret_cast<uint4*>(page + ((off >> 3) * NCH + ch) * 128 + (off & 7) * 16);
        if constexpr (E == 2) {
            *dst = first ? a0 : __ldg(reinterpret_cast<const uint4*>(src + ch * 16));
        } else {
            const float sc = (which ? v_scales : k_scales)[(size_t)blk * Hkv + g];
            const uint4 a = first ? a0 : __ldg(reinterpret_cast<const uint4*>(src + ch * 32));
            const uint4 b = first ? b0 : __ldg(reinterpret_cast<const uint4*>(src + ch * 32 + 16));
            const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
            uint32_t packed[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t word = 0;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint32_t x = w[2 * j + h];
                    const float lo = __fdiv_rn(bf16_lo(x), sc), hi = __fdiv_rn(bf16_hi(x), sc);
                    const uint32_t c0 = __nv_cvt_float_to_fp8(lo, __NV_SATFINITE, __NV_E4M3);
                    const uint32_t c1 = __nv_cvt_float_to_fp8(hi, __NV_SATFINITE, __NV_E4M3);
                    word |= (c0 | (c1 << 8)) << (16 * h);
                }
                packed[j] = word;
            }
            *dst = make_uint4(packed[0], packed[1], packed[2], packed[3]);
        }
    }
}

// Copy-on-write of whole blocks: pairs[2i] -> pairs[2i + 1], every kv-head's
// K and V page (16-byte chunks, one per thread), and the FP8 scales.
__global__ void __launch_bounds__(256) copy_blocks_kernel(const int32_t* __restrict__ pairs, int n, int Hkv,
                                                          int page_chunks, int64_t num_blocks, uint8_t* k_cache,
                                                          uint8_t* v_cache, float* k_scales, float* v_scales) {
    griddep_launch();
    griddep_wait();                              // the previous kernel's reads of these pages are done
    const int64_t per_pair = (int64_t)2 * Hkv * page_chunks;
    const int64_t total = (int64_t)n * per_pair;
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int i = (int)(idx / per_pair);
        const int64_t rem = idx % per_pair;
        const int which = (int)(rem / ((int64_t)Hkv * page_chunks));      // 0 = K, 1 = V
        const int64_t within = rem % ((int64_t)Hkv * page_chunks);       // (head, chunk) of the block
        const int32_t src = pairs[2 * i], dst = pairs[2 * i + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) continue;
        uint8_t* base = which ? v_cache : k_cache;
        const size_t blk_bytes = (size_t)Hkv * page_chunks * 16;
        const uint4 x = *reinterpret_cast<const uint4*>(base + (size_t)src * blk_bytes + within * 16);
        *reinterpret_cast<uint4*>(base + (size_t)dst * blk_bytes + within * 16) = x;
        float* sc = which ? v_scales : k_scales;
        if (sc && within % page_chunks == 0) {           // the head's first chunk also copies its scale
            const int64_t head = within / page_chunks;
            sc[(size_t)dst * Hkv + head] = sc[(size_t)src * Hkv + head];
        }
    }
}

cudaError_t launch_copy_blocks(const pkv_cache& c, const int32_t* pairs, int n, float* k_scales, float* v_scales,
                               cudaStream_t st, int num_sms) {
    const int E = c.kv_dtype == PKV_KV_FP8_E4M3 ? 1 : 2;
    const int page_chunks = kBlock * c.head_dim * E / 16;
    const int64_t total = (int64_t)n * 2 * c.num_kv_heads * page_chunks;
    int64_t blocks = (total + 255) / 256;
    if (blocks > (int64_t)num_sms * 8) blocks = (int64_t)num_sms * 8;
    if (blocks < 1) blocks = 1;
    return launch_pdl(copy_blocks_kernel, dim3((unsigned)blocks), dim3(256), 0, st, pairs, n, (int)c.num_kv_heads,
                      page_chunks, (int64_t)c.num_blocks, (uint8_t*)c.k_cache, (uint8_t*)c.v_cache,
                      E == 1 ? k_scales : (float*)nullptr, E == 1 ? v_scales : (float*)nullptr);
}

cudaError_t launch_append(const pkv_cache& c, const void* k_new, const void* v_new, const int64_t* slots,
                          int64_t num_tokens, int* err, cudaStream_t st, int num_sms) {
    const int E = c.kv_dtype == PKV_KV_FP8_E4M3 ? 1 : 2;
    const int64_t total = num_tokens * c.num_kv_heads * (c.head_dim * E / 16) * 2;
    // a decode step's few bf16 tokens: 32-thread CTAs, one chunk a thread (one of them fits
    // beside each resident attention CTA); FP8 (whose encode divides every value) and larger
    // appends (a prefill's prompt): 256-thread CTAs, up to 8 per SM
    const bool small = E == 2 && total <= (int64_t)num_sms * 32 * 2;
    const int threads = small ? 32 : 256;
    int64_t blocks = (total + threads - 1) / threads;
    const int64_t cap = (int64_t)num_sms * (small ? 2 : 8);
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    // A programmatic dependent launch: the kernel may be scheduled while the
    // previous one (an attention that triggers early) still runs, and waits
    // for it before touching memory.
    const float* ks = E == 2 ? nullptr : c.k_scales;
    const float* vs = E == 2 ? nullptr : c.v_scales;
    return launch_pdl(E == 2 ? append_kernel<2> : append_kernel<1>, dim3((unsigned)blocks), dim3(threads), 0, st,
                      (const uint8_t*)k_new, (const uint8_t*)v_new, slots, num_tokens, (int)c.num_kv_heads,
                      (int)c.head_dim, (int64_t)c.num_blocks, (uint8_t*)c.k_cache, (uint8_t*)c.v_cache, ks, vs, err);
}

}  // namespace pkv
