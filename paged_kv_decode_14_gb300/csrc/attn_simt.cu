// Paged decode / verify attention on CUDA cores (FP32 FMA), one warp per page.
//
// Computes, for every (sequence b, kv-head g), the GQA group's rows
// r = i * G + hl (query i of the window, query head g * G + hl):
//   out_r = softmax_j(scale * q_r . k_j) v_j over positions j <= L - Q + i
// (the paged attention of the inferd and lfm25-inference READMEs), with the
// group folded into one CTA so each page is read once per row pass.
//
// Grid: a persistent set of CTAs over the balanced page partition of
// common.cuh.  Each CTA walks its pieces; its 4 warps take the pages of a
// piece round robin, staging each (K, V) page pair in shared memory with
// 16-byte cp.async (double-buffered per warp), and keep an online softmax
// state (running max m, sum l, accumulator) per row.  At the end of a piece the
// warps' states are combined; complete segments are written as bf16, cut
// segments leave a partial and the last CTA of the segment merges.
#include "common.cuh"

namespace pkv {
namespace simt {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;

template <int D, int E, int RT>
struct Cfg {
    static constexpr int NCH = D * E / 16;        // 16-byte chunks per token
    static constexpr int C = 16 / E;              // elements per chunk
    static constexpr int PAGE = kBlock * D * E;   // bytes per page
    static constexpr int DPL = D / 32;            // PV: dims per lane
    static constexpr int QS = D + 4;              // padded q row stride (floats)
    static constexpr int VEC = PAGE / 16 / 32;    // 16-byte copies per lane per page
    // shared memory layout (bytes)
    static constexpr int OFF_PAGES = 0;                                   // [warp][buf][K|V][PAGE]
    static constexpr int OFF_Q = OFF_PAGES + kWarps * 2 * 2 * PAGE;       // float [RT][QS]
    static constexpr int OFF_P = OFF_Q + RT * QS * 4;                     // float [warp][RT][16]
    static constexpr int OFF_CMB = OFF_P + kWarps * RT * 16 * 4;          // float [warp][RT][D+2]
    static constexpr int SMEM = OFF_CMB + kWarps * RT * (D + 2) * 4;
};

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

// q . chunk for one 16-byte chunk of a token (C elements) against C floats of q.
template <int E>
__device__ __forceinline__ float chunk_dot(const uint4 w, const float* q) {
    const uint32_t v[4] = {w.x, w.y, w.z, w.w};
    float acc = 0.f;
    if constexpr (E == 2) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 qq = *reinterpret_cast<const float2*>(q + 2 * j);
            acc = fmaf(bf16_lo(v[j]), qq.x, acc);
            acc = fmaf(bf16_hi(v[j]), qq.y, acc);
        }
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 a = e4m3x2_to_float2(v[j]);
            const float2 b = e4m3x2_to_float2(v[j] >> 16);
            const float4 qq = *reinterpret_cast<const float4*>(q + 4 * j);
            acc = fmaf(a.x, qq.x, acc);
            acc = fmaf(a.y, qq.y, acc);
            acc = fmaf(b.x, qq.z, acc);
            acc = fmaf(b.y, qq.w, acc);
        }
    }
    return acc;
}

// DPL consecutive elements of a token row starting at the lane's first dim.
template <int E, int DPL>
__device__ __forceinline__ void load_v(const uint8_t* addr, float (&v)[DPL]) {
    if constexpr (E == 2) {
        if constexpr (DPL == 4) {
            const uint2 w = *reinterpret_cast<const uint2*>(addr);
            v[0] = bf16_lo(w.x); v[1] = bf16_hi(w.x); v[2] = bf16_lo(w.y); v[3] = bf16_hi(w.y);
        } else {
            const uint32_t w = *reinterpret_cast<const uint32_t*>(addr);
            v[0] = bf16_lo(w); v[1] = bf16_hi(w);
        }
    } else {
        if constexpr (DPL == 4) {
            const uint32_t w = *reinterpret_cast<const uint32_t*>(addr);
            const float2 a = e4m3x2_to_float2(w), b = e4m3x2_to_float2(w >> 16);
            v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
        } else {
            const uint32_t w = *reinterpret_cast<const uint16_t*>(addr);
            const float2 a = e4m3x2_to_float2(w);
            v[0] = a.x; v[1] = a.y;
        }
    }
}

template <int D, int E, int RT>
__global__ void __launch_bounds__(kThreads) attn_simt_kernel(const AttnParams p) {
    using K = Cfg<D, E, RT>;
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int scratch[kThreads / 32 + 1];
    __shared__ int s_ticket;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cta = blockIdx.x;
    griddep_launch();     // the next kernel on the stream may launch (it waits for this grid's results)
    griddep_wait();       // inputs of the previous kernel on the stream are visible
    Cursor cur;
    int u0, u1, W, P;
    if (!plan_locate<kThreads>(p, cta, gridDim.x, scratch, &cur, &u0, &u1, &W, &P)) return;
    const int ncta = P;

    float* qs = reinterpret_cast<float*>(smem + K::OFF_Q);
    float* pb = reinterpret_cast<float*>(smem + K::OFF_P) + warp * RT * 16;
    float* cmb = reinterpret_cast<float*>(smem + K::OFF_CMB);
    uint8_t* wpages = smem + K::OFF_PAGES + warp * 2 * 2 * K::PAGE;
    const int G = p.group, Hkv = p.num_kv_heads;

    int u = u0;
    while (u < u1) {
        const int g = (u - cur.Ub) / cur.nb;
        const int S0 = cur.Ub + g * cur.nb, S1 = S0 + cur.nb;
        const int pe = min(u1, S1);
        const int pg0 = u - S0, pg1 = pe - S0;        // pages [pg0, pg1) of segment
        const int npg = pg1 - pg0;
        const int R = G * cur.Q;
        const int L = cur.L, lim0 = cur.L - cur.Q;
        const int32_t* table = p.block_tables + (size_t)cur.b * p.max_blocks_per_seq;
        const bool complete = (S0 >= u0) && (S1 <= u1);
        float* slot = complete ? nullptr : slot_ptr(p, cta, S0, u0);

        for (int row0 = 0; row0 < R; row0 += RT) {
            // q rows of this pass -> shared (fp32)
            __syncthreads();
            for (int idx = tid; idx < RT * D; idx += kThreads) {
                const int r = idx / D, d = idx % D, rr = row0 + r;
                float v = 0.f;
                if (rr < R) {
                    const int i = rr / G, hl = rr % G;
                    v = __bfloat162float(p.q[((size_t)(cur.qoff + i) * p.num_q_heads + g * G + hl) * D + d]);
                }
                qs[r * K::QS + d] = v;
            }
            __syncthreads();

            float m[RT], l[RT], acc[RT][K::DPL];
#pragma unroll
            for (int r = 0; r < RT; ++r) {
                m[r] = -INFINITY;
                l[r] = 0.f;
#pragma unroll
                for (int j = 0; j < K::DPL; ++j) acc[r][j] = 0.f;
            }

            // issue page `lp` (local index) of this warp into buffer `buf`
            auto issue = [&](int lp, int buf) {
                int blk = table[pg0 + lp];
                if (blk < 0 || blk >= p.num_blocks) {
                    raise_error(p.err, PKV_DEVERR_BLOCK_ID);
                    blk = 0;
                }
                const size_t page_off = ((size_t)blk * p.cache_kv_heads + cache_head(p, g)) * K::PAGE;
                uint8_t* dk = wpages + buf * 2 * K::PAGE;
                uint8_t* dv = dk + K::PAGE;
#pragma unroll
                for (int j = 0; j < K::VEC; ++j) {
                    const int o = (j * 32 + lane) * 16;
                    cp_async16(dk + o, p.k_cache + page_off + o);
                    cp_async16(dv + o, p.v_cache + page_off + o);
                }
            };

            int buf = 0;
            if (warp < npg) issue(warp, 0);
            cp_async_commit();
            for (int lp = warp; lp < npg; lp += kWarps) {
                if (lp + kWarps < npg) issue(lp + kWarps, buf ^ 1);
                cp_async_commit();
                cp_async_wait<1>();
                __syncwarp();
                const uint8_t* kp = wpages + buf * 2 * K::PAGE;
                const uint8_t* vp = kp + K::PAGE;
                const int blk_raw = table[pg0 + lp];
                const int blk = (blk_raw < 0 || blk_raw >= p.num_blocks) ? 0 : blk_raw;
                float ksc = p.scale_log2, vsc = 1.f;
                if constexpr (E == 1) {
                    ksc *= p.k_scales[(size_t)blk * p.cache_kv_heads + cache_head(p, g)];
                    vsc = p.v_scales[(size_t)blk * p.cache_kv_heads + cache_head(p, g)];
                }
                const int tok0 = (pg0 + lp) * kBlock;

                // ---- S = q . k for (row, token) pairs: pair = lane + 32 k
                const int t = lane & 15, half = lane >> 4;
                float s[RT / 2];
#pragma unroll
                for (int k = 0; k < RT / 2; ++k) {
                    const int r = 2 * k + half;
                    const float* qrow = qs + r * K::QS;
                    float dot = 0.f;
#pragma unroll
                    for (int ch = 0; ch < K::NCH; ++ch) {
                        const uint4 w = *reinterpret_cast<const uint4*>(kp + ((t >> 3) * K::NCH + ch) * 128 + (t & 7) * 16);
                        dot += chunk_dot<E>(w, qrow + ch * K::C);
                    }
                    const int rr = row0 + r, pos = tok0 + t;
                    const bool vis = rr < R && pos < L && pos <= lim0 + rr / G;
                    s[k] = vis ? dot * ksc : -INFINITY;
                }
                // ---- online softmax per row (rows 2k live on lanes 0-15, 2k+1 on 16-31)
                float alpha[RT];
#pragma unroll
                for (int k = 0; k < RT / 2; ++k) {
                    float mx = s[k];
#pragma unroll
                    for (int o = 8; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                    const float mx0 = __shfl_sync(0xffffffffu, mx, 0), mx1 = __shfl_sync(0xffffffffu, mx, 16);
                    const float mn0 = fmaxf(m[2 * k], mx0), mn1 = fmaxf(m[2 * k + 1], mx1);
                    const float mown = half ? mn1 : mn0;
                    const float pv = (s[k] == -INFINITY) ? 0.f : exp2f(s[k] - mown);
                    pb[(2 * k + half) * 16 + t] = pv * vsc;
                    float ps = pv;
#pragma unroll
                    for (int o = 8; o >= 1; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
                    const float ps0 = __shfl_sync(0xffffffffu, ps, 0), ps1 = __shfl_sync(0xffffffffu, ps, 16);
                    const float a0 = (m[2 * k] == -INFINITY) ? 0.f : exp2f(m[2 * k] - mn0);
                    const float a1 = (m[2 * k + 1] == -INFINITY) ? 0.f : exp2f(m[2 * k + 1] - mn1);
                    l[2 * k] = l[2 * k] * a0 + ps0;
                    l[2 * k + 1] = l[2 * k + 1] * a1 + ps1;
                    m[2 * k] = mn0;
                    m[2 * k + 1] = mn1;
                    alpha[2 * k] = a0;
                    alpha[2 * k + 1] = a1;
                }
                __syncwarp();
                // ---- acc = acc * alpha + P V ; the lane owns dims [lane*DPL, lane*DPL + DPL)
                const int lb = lane * K::DPL * E;         // byte offset within a token row
                const int ch = lb >> 4, within = lb & 15;
#pragma unroll
                for (int r = 0; r < RT; ++r)
#pragma unroll
                    for (int j = 0; j < K::DPL; ++j) acc[r][j] *= alpha[r];
#pragma unroll 4
                for (int step = 0; step < kBlock; ++step) {
                    const int tau = (step + ch) & 15;
                    float v[K::DPL];
                    load_v<E, K::DPL>(vp + ((tau >> 3) * K::NCH + ch) * 128 + (tau & 7) * 16 + within, v);
                    if (tok0 + tau >= L) {          // unwritten tail slots may hold NaN
#pragma unroll
                        for (int j = 0; j < K::DPL; ++j) v[j] = 0.f;
                    }
#pragma unroll
                    for (int r = 0; r < RT; ++r) {
                        const float pr = pb[r * 16 + tau];
#pragma unroll
                        for (int j = 0; j < K::DPL; ++j) acc[r][j] = fmaf(pr, v[j], acc[r][j]);
                    }
                }
                __syncwarp();
                buf ^= 1;
            }
            cp_async_wait<0>();

            // ---- combine the 4 warps' states
            float* mine = cmb + warp * RT * (D + 2);
            if (lane == 0) {
#pragma unroll
                for (int r = 0; r < RT; ++r) {
                    mine[r] = m[r];
                    mine[RT + r] = l[r];
                }
            }
#pragma unroll
            for (int r = 0; r < RT; ++r)
#pragma unroll
                for (int j = 0; j < K::DPL; ++j) mine[2 * RT + r * D + lane * K::DPL + j] = acc[r][j];
            __syncthreads();
            for (int idx = tid; idx < RT * D; idx += kThreads) {
                const int r = idx / D, d = idx % D, rr = row0 + r;
                if (rr >= R) continue;
                float M = -INFINITY;
#pragma unroll
                for (int w = 0; w < kWarps; ++w) M = fmaxf(M, cmb[w * RT * (D + 2) + r]);
                float den = 0.f, num = 0.f;
#pragma unroll
                for (int w = 0; w < kWarps; ++w) {
                    const float* st = cmb + w * RT * (D + 2);
                    const float sc = (st[r] == -INFINITY) ? 0.f : exp2f(st[r] - M);
                    den += sc * st[RT + r];
                    num += sc * st[2 * RT + r * D + d];
                }
                if (complete) {
                    const int i = rr / G, hl = rr % G;
                    p.out[((size_t)(cur.qoff + i) * p.num_q_heads + g * G + hl) * D + d] = __float2bfloat16_rn(num / den);
                } else {
                    if (d == 0) {
                        slot[rr] = M;
                        slot[p.rows_pad + rr] = den;
                    }
                    slot[2 * p.rows_pad + (size_t)rr * D + d] = num;
                }
            }
        }

        if (!complete) {
            // ticket: the last CTA of the segment merges its partials
            __threadfence();
            __syncthreads();
            if (tid == 0) {
                const int need = owner_cta(S1 - 1, W, ncta) - owner_cta(S0, W, ncta) + 1;
                const int old = atomicAdd(p.tickets + cur.b * Hkv + g, 1);
                s_ticket = (old == need - 1);
                if (s_ticket) p.tickets[cur.b * Hkv + g] = 0;
            }
            __syncthreads();
            if (s_ticket) {
                __threadfence();
                merge_segment<kThreads>(p, cur, g, S0, S1, W, ncta, D);
            }
        }

        u = pe;
        if (u < u1 && u == cur.Ub + cur.nb * Hkv) cursor_next(p, cur);
    }
}

}  // namespace simt

// ------------------------------------------------------------------ launch

template <int D, int E, int RT>
static cudaError_t launch_simt_t(const AttnParams& p, int ncta, cudaStream_t st) {
    using K = simt::Cfg<D, E, RT>;
    static std::atomic<uint64_t> attr_set{0};
    return launch_pdl_bigsmem(attr_set, simt::attn_simt_kernel<D, E, RT>, dim3(ncta), dim3(simt::kThreads),
                              (size_t)K::SMEM, st, p);
}

template <int D, int E>
static cudaError_t launch_simt_d(const AttnParams& p, int ncta, cudaStream_t st) {
    if (p.rows <= 4) return launch_simt_t<D, E, 4>(p, ncta, st);
    if (p.rows <= 8) return launch_simt_t<D, E, 8>(p, ncta, st);
    return launch_simt_t<D, E, 16>(p, ncta, st);
}

cudaError_t launch_attention_simt(const AttnParams& p, int head_dim, int elem_bytes, int ncta,
                                  cudaStream_t st) {
    if (head_dim == 128) return elem_bytes == 2 ? launch_simt_d<128, 2>(p, ncta, st) : launch_simt_d<128, 1>(p, ncta, st);
    return elem_bytes == 2 ? launch_simt_d<64, 2>(p, ncta, st) : launch_simt_d<64, 1>(p, ncta, st);
}

int simt_rows_pad(int rows) { return rows <= 4 ? 4 : rows <= 8 ? 8 : ((rows + 15) / 16) * 16; }

}  // namespace pkv
