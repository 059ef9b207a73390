// Fused rotary position embedding + paged_kv_append, and FP8 scales chosen
// at append time (the lfm25-inference file list: kernels/rope.cu,
// kernels/kv_cache.cu).  Contract: include/pagedkv.h, pkv_paged_kv_append_rope.
//
// Rotation (rotate-half form): for a row x of head_dim D at position p and
// i < D/2, with a_i = p * theta^(-2i/D),
//   y_i = x_i cos a_i - x_{i+D/2} sin a_i,  y_{i+D/2} = x_{i+D/2} cos a_i + x_i sin a_i,
// evaluated in fp64 (a token's CTA computes its D/2 angles once, in fp64, so
// large positions keep their precision) and rounded once to bf16.
//
// FP8 scales from the values: for every (block, kv-head) whose offset-0
// slot this call writes, scale = max |value| over the call's values in that
// block and head (NaN ignored) / 448 in IEEE fp32, 1 if that maximum is 0.
// Three launches in stream order: mark those scales (the bits of -0.0),
// raise them to (sign bit | |value| bits) with integer atomicMax (a float's
// magnitude orders like its bits), then encode, turning a marked scale into
// absmax / 448 (the offset-0 token's thread stores it).
#include "common.cuh"

namespace pkv {
namespace rope {

constexpr int kThreads = 256;
constexpr int kMaxHalf = 64;                      // head_dim <= 128
constexpr uint32_t kMark = 0x80000000u;

// cos / sin of the token's D/2 angles into shared memory (threads i < D/2).
__device__ __forceinline__ void angles(double2* cs, int D, int pos, double theta) {
    const int half = D / 2;
    for (int i = threadIdx.x; i < half; i += blockDim.x) {
        const double inv = pow(theta, -2.0 * (double)i / (double)D);
        double s, c;
        sincos((double)pos * inv, &s, &c);
        cs[i] = make_double2(c, s);
    }
}

// Rotated pair (i, i + D/2) of one bf16 row, rounded to bf16.
__device__ __forceinline__ void rotate_pair(const __nv_bfloat16* row, int i, int half, double2 cs, __nv_bfloat16& lo,
                                            __nv_bfloat16& hi) {
    const double a = (double)__bfloat162float(row[i]), b = (double)__bfloat162float(row[i + half]);
    lo = __double2bfloat16(a * cs.x - b * cs.y);
    hi = __double2bfloat16(b * cs.x + a * cs.y);
}

__device__ __forceinline__ bool slot_block(int64_t s, int64_t num_blocks, int64_t& blk, int& off) {
    if (s < 0 || s / kBlock >= num_blocks) return false;
    blk = s / kBlock;
    off = (int)(s % kBlock);
    return true;
}

// Mark the scales of the blocks this call starts (one thread per token and kv-head).
__global__ void __launch_bounds__(kThreads) mark_kernel(const int64_t* __restrict__ slots, int64_t T, int Hkv,
                                                        int64_t num_blocks, uint32_t* k_scales, uint32_t* v_scales) {
    griddep_launch();
    griddep_wait();
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < T * Hkv;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = idx / Hkv;
        const int g = (int)(idx % Hkv);
        int64_t blk;
        int off;
        if (!slot_block(slots[t], num_blocks, blk, off) || off != 0) continue;
        k_scales[blk * Hkv + g] = kMark;
        v_scales[blk * Hkv + g] = kMark;
    }
}

// Raise the marked scales to the call's |value| maxima (one CTA per token,
// one warp per kv-head at a time).
__global__ void __launch_bounds__(kThreads) absmax_kernel(const __nv_bfloat16* __restrict__ k_new,
                                                          const __nv_bfloat16* __restrict__ v_new,
                                                          const int64_t* __restrict__ slots,
                                                          const int32_t* __restrict__ positions, double theta,
                                                          int Hkv, int D, int64_t num_blocks, uint32_t* k_scales,
                                                          uint32_t* v_scales) {
    __shared__ double2 cs[kMaxHalf];
    griddep_launch();
    griddep_wait();
    const int64_t t = blockIdx.x;
    int64_t blk;
    int off;
    if (!slot_block(slots[t], num_blocks, blk, off)) return;        // (uniform over the CTA)
    const int half = D / 2;
    if (positions) {
        angles(cs, D, positions[t], theta);
        __syncthreads();
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int g = warp; g < Hkv; g += kThreads / 32) {
        const size_t base = ((size_t)t * Hkv + g) * D;
        float mk = 0.f, mv = 0.f;
        for (int i = lane; i < half; i += 32) {
            float a, b;
            if (positions) {
                __nv_bfloat16 lo, hi;
                rotate_pair(k_new + base, i, half, cs[i], lo, hi);
                a = __bfloat162float(lo);
                b = __bfloat162float(hi);
            } else {
                a = __bfloat162float(k_new[base + i]);
                b = __bfloat162float(k_new[base + i + half]);
            }
            mk = fmaxf(mk, fmaxf(fabsf(a), fabsf(b)));                // (fmaxf ignores NaN)
            mv = fmaxf(mv, fmaxf(fabsf(__bfloat162float(v_new[base + i])), fabsf(__bfloat162float(v_new[base + i + half]))));
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            mk = fmaxf(mk, __shfl_xor_sync(0xffffffffu, mk, o));
            mv = fmaxf(mv, __shfl_xor_sync(0xffffffffu, mv, o));
        }
        if (lane == 0) {
            uint32_t* kp = k_scales + blk * Hkv + g;
            uint32_t* vp = v_scales + blk * Hkv + g;
            // only scales this call marked: a marked value keeps its sign bit
            if (*reinterpret_cast<volatile uint32_t*>(kp) & kMark) atomicMax(kp, kMark | __float_as_uint(mk));
            if (*reinterpret_cast<volatile uint32_t*>(vp) & kMark) atomicMax(vp, kMark | __float_as_uint(mv));
        }
    }
}

// The scale this token encodes with: a marked scale becomes absmax / 448
// (the offset-0 token stores it; any token reading either value computes the
// same number).
__device__ __forceinline__ float final_scale(uint32_t* sp, bool owner) {
    const uint32_t bits = *reinterpret_cast<volatile uint32_t*>(sp);
    if (!(bits & kMark)) return __uint_as_float(bits);
    const float amax = __uint_as_float(bits & ~kMark);
    const float s = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
    if (owner) *reinterpret_cast<volatile uint32_t*>(sp) = __float_as_uint(s);
    return s;
}

// One CTA per token: rotate its q rows in place, its K rows into shared
// memory, then store K and V into the token's slot (bf16 copy, or E4M3 encode
// with the page's scale).
template <int E, bool AUTOSCALE>
__global__ void __launch_bounds__(kThreads) rope_append_kernel(
    const __nv_bfloat16* __restrict__ k_new, const __nv_bfloat16* __restrict__ v_new, const int64_t* __restrict__ slots,
    const int32_t* __restrict__ positions, double theta, __nv_bfloat16* q, int Hq, int Hkv, int D, int64_t num_blocks,
    uint8_t* k_cache, uint8_t* v_cache, float* k_scales, float* v_scales, int* err) {
    extern __shared__ __align__(16) uint8_t rope_smem[];
    __shared__ double2 cs[kMaxHalf];
    __shared__ float sc[2][32];                         // this token's (K, V) scale per kv-head (FP8)
    // No early trigger here: this kernel rotates q in place, and the attention that follows reads
    // its q rows before its own dependency wait, so it may launch only once this grid has ended.
    griddep_wait();
    const int64_t t = blockIdx.x;
    const int half = D / 2, tid = threadIdx.x;
    if (positions) angles(cs, D, positions[t], theta);
    __syncthreads();
    // q rows of the token, in place
    if (q && positions) {
        for (int idx = tid; idx < Hq * half; idx += kThreads) {
            const int h = idx / half, i = idx % half;
            __nv_bfloat16* row = q + ((size_t)t * Hq + h) * D;
            __nv_bfloat16 lo, hi;
            rotate_pair(row, i, half, cs[i], lo, hi);
            row[i] = lo;
            row[i + half] = hi;
        }
    }
    int64_t blk;
    int off;
    if (!slot_block(slots[t], num_blocks, blk, off)) {
        if (slots[t] >= 0 && tid == 0) raise_error(err, PKV_DEVERR_SLOT);
        return;
    }
    // K rows, rotated, into shared memory
    __nv_bfloat16* kr = reinterpret_cast<__nv_bfloat16*>(rope_smem);      // [Hkv][D]
    for (int idx = tid; idx < Hkv * half; idx += kThreads) {
        const int g = idx / half, i = idx % half;
        const __nv_bfloat16* row = k_new + ((size_t)t * Hkv + g) * D;
        if (positions) {
            __nv_bfloat16 lo, hi;
            rotate_pair(row, i, half, cs[i], lo, hi);
            kr[g * D + i] = lo;
            kr[g * D + i + half] = hi;
        } else {
            kr[g * D + i] = row[i];
            kr[g * D + i + half] = row[i + half];
        }
    }
    if constexpr (E == 1) {
        for (int idx = tid; idx < 2 * Hkv; idx += kThreads) {
            const int which = idx / Hkv, g = idx % Hkv;
            float* sp = (which ? v_scales : k_scales) + blk * Hkv + g;
            sc[which][g] = AUTOSCALE ? final_scale(reinterpret_cast<uint32_t*>(sp), off == 0) : *sp;
        }
    }
    __syncthreads();
    // store: one thread per (kv-head, 16-byte cache chunk, K|V)
    const int NCH = D * E / 16;
    for (int idx = tid; idx < Hkv * NCH * 2; idx += kThreads) {
        const int which = idx & 1, rem = idx >> 1, g = rem / NCH, ch = rem % NCH;
        const __nv_bfloat16* src = which ? v_new + ((size_t)t * Hkv + g) * D : kr + g * D;
        uint8_t* page = (which ? v_cache : k_cache) + ((size_t)blk * Hkv + g) * (size_t)(kBlock * D * E);
        uint4* dst = reinterpret_cast<uint4*>(page + ((off >> 3) * NCH + ch) * 128 + (off & 7) * 16);
        if constexpr (E == 2) {
            const uint16_t* s16 = reinterpret_cast<const uint16_t*>(src) + ch * 8;
            uint32_t w[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) w[j] = (uint32_t)s16[2 * j] | ((uint32_t)s16[2 * j + 1] << 16);
            *dst = make_uint4(w[0], w[1], w[2], w[3]);
        } else {
            const float s = sc[which][g];
            uint32_t packed[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t word = 0;
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const float x = __bfloat162float(src[ch * 16 + 4 * j + h]);
                    word |= (uint32_t)__nv_cvt_float_to_fp8(__fdiv_rn(x, s), __NV_SATFINITE, __NV_E4M3) << (8 * h);
                }
                packed[j] = word;
            }
            *dst = make_uint4(packed[0], packed[1], packed[2], packed[3]);
        }
    }
}

}  // namespace rope

cudaError_t launch_append_rope(const pkv_cache& c, const void* k_new, const void* v_new, const int64_t* slots,
                               int64_t T, const int32_t* positions, double theta, void* q, int Hq, bool autoscale,
                               int* err, cudaStream_t st, int num_sms) {
    using namespace rope;
    const int E = c.kv_dtype == PKV_KV_FP8_E4M3 ? 1 : 2;
    const int Hkv = c.num_kv_heads, D = c.head_dim;
    const size_t smem = (size_t)Hkv * D * 2;
    const auto* kb = (const __nv_bfloat16*)k_new;
    const auto* vb = (const __nv_bfloat16*)v_new;
    float* ks = const_cast<float*>(c.k_scales);
    float* vs = const_cast<float*>(c.v_scales);
    cudaError_t e = cudaSuccess;
    if (E == 1 && autoscale) {
        int64_t blocks = (T * Hkv + kThreads - 1) / kThreads;
        if (blocks > (int64_t)num_sms * 8) blocks = (int64_t)num_sms * 8;
        e = launch_pdl(mark_kernel, dim3((unsigned)blocks), dim3(kThreads), 0, st, slots, T, Hkv, (int64_t)c.num_blocks,
                       (uint32_t*)ks, (uint32_t*)vs);
        if (e != cudaSuccess) return e;
        e = launch_pdl(absmax_kernel, dim3((unsigned)T), dim3(kThreads), 0, st, kb, vb, slots, positions, theta, Hkv, D,
                       (int64_t)c.num_blocks, (uint32_t*)ks, (uint32_t*)vs);
        if (e != cudaSuccess) return e;
    }
    auto* qb = (__nv_bfloat16*)q;
    auto* kc = (uint8_t*)c.k_cache;
    auto* vc = (uint8_t*)c.v_cache;
    if (E == 2)
        return launch_pdl(rope_append_kernel<2, false>, dim3((unsigned)T), dim3(kThreads), smem, st, kb, vb, slots,
                          positions, theta, qb, Hq, Hkv, D, (int64_t)c.num_blocks, kc, vc, ks, vs, err);
    return autoscale ? launch_pdl(rope_append_kernel<1, true>, dim3((unsigned)T), dim3(kThreads), smem, st, kb, vb,
                                  slots, positions, theta, qb, Hq, Hkv, D, (int64_t)c.num_blocks, kc, vc, ks, vs, err)
                     : launch_pdl(rope_append_kernel<1, false>, dim3((unsigned)T), dim3(kThreads), smem, st, kb, vb,
                                  slots, positions, theta, qb, Hq, Hkv, D, (int64_t)c.num_blocks, kc, vc, ks, vs, err);
}

}  // namespace pkv
