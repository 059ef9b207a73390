// Paged decode / verify attention on the 5th-generation tensor cores
// (tcgen05 MMA, accumulators in TMEM, pages staged by 1-D bulk copies).
//
// Computes what attn_simt.cu computes (the paged GQA/XQA attention of the
// lfm25-inference README, equal to dense attention per the inferd
// equivalence gate): for every (sequence b, kv-head g), rows r = i*G + hl,
//   out_r = softmax_j(scale * q_r . k_j) v_j,  j <= L - Q + i.
//
// Work partition and merge: the balanced page partition of common.cuh, one
// persistent CTA per SM.  A CTA streams its pages in tiles of 8 pages = 128
// tokens.  Per tile:
//   S^T[128 tok, N] = K_tile[128 tok, D] . Q^T[D, N]       (MMA, M=128, K-major A and B)
//   softmax on S^T rows (one thread per token, TMEM lane = token)
//   O^T[128 d, N]   = V_tile^T[d, 128 tok] . P^T[128 tok, N] (MMA, M=128, MN-major A and B)
//   correction acc = acc * alpha + O^T (one thread per head-dim row)
// with N = 16 or 32 columns holding the group's R = G*Q query rows.  The
// query group sits on the MMA's N side ("swap AB"), so G*Q rows of 4..32 do
// not waste a 64/128-row M tile.  When 2R <= 16, P is split into a bf16 high
// part and a bf16 low part on adjacent columns (free: N is 16 anyway), so the
// P.V product keeps about 16 bits of P.
//
// The cache's page layout (16-byte chunks, core matrices of 8 tokens x 16
// bytes, see pagedkv.h) is exactly the tensor core's no-swizzle canonical
// layout: K pages are K-major A operands and V pages MN-major A operands as
// copied, so a page goes HBM -> shared memory in one bulk copy and is never
// touched by the CUDA cores (except zeroing the unwritten tail rows of a
// sequence's last page, which may hold NaN).
//
// Warp roles (192 threads): warps 0-3 softmax + correction + epilogue (their
// TMEM lane quarters), warp 4 producer (bulk copies, q staging), warp 5 MMA
// issuer.  Every mbarrier wait is bounded (2 s); a timeout sets
// PKV_DEVERR_TIMEOUT and an abort flag, all roles wind down, in-flight copies
// are drained and TMEM is freed before the CTA exits.
#include "common.cuh"
#include "tc_ptx.cuh"

namespace pkv {
namespace tc {

using namespace ptx;

constexpr int kTP = 8;                        // pages per tile
constexpr int kTileTok = kTP * kBlock;        // 128 tokens = MMA M
constexpr int kThreads = 192;
constexpr int kProducerWarp = 4, kMmaWarp = 5;
constexpr int kSoftThreads = 128;
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr int kMaxSmem = 232448;

template <int D, int NPAD, bool SPLIT, int NS>
struct Cfg {
    static constexpr int PAGE = kBlock * D * 2;
    static constexpr int NCH = D / 8;                   // 16-byte chunks per token row
    static constexpr int TILE = kTP * PAGE;
    static constexpr int VSLACK = D == 64 ? 1024 : 0;   // M=128 PV on D=64 reads 1 KiB past a page
    static constexpr int OFF_K = 0;                     // + st * TILE
    static constexpr int OFF_V = NS * TILE;             // + st * (TILE + VSLACK)
    static constexpr int OFF_Q = OFF_V + NS * (TILE + VSLACK);
    static constexpr int QBUF = NPAD * D * 2;
    static constexpr int OFF_P = OFF_Q + 2 * QBUF;
    static constexpr int PBUF = NPAD * kTileTok * 2;
    static constexpr int OFF_RED = OFF_P + 2 * PBUF;             // float [2][4][RMAX]
    static constexpr int RMAX = SPLIT ? NPAD / 2 : NPAD;         // query rows per (b, g)
    static constexpr int OFF_LRED = OFF_RED + 2 * 4 * RMAX * 4;  // float [4][RMAX]
    static constexpr int OFF_BAR = OFF_LRED + 4 * RMAX * 4;
    static constexpr int NBAR = 3 * NS + 11;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;          // tmem addr, abort, ticket, zero
    static constexpr int SMEM_USED = OFF_MISC + 16 + 128;        // + base alignment slack
    // One CTA per SM either way: take the whole per-block budget, so every
    // operand read the descriptors can form stays inside the allocation.
    static constexpr int SMEM = kMaxSmem - 1024;
    static constexpr int TMEM_COLS = 4 * NPAD;                   // S[2], O[2]
    static_assert(SMEM_USED <= SMEM, "shared memory budget");
    static_assert(TMEM_COLS >= 32 && (TMEM_COLS & (TMEM_COLS - 1)) == 0, "TMEM allocation size");
};

// barrier indices
template <int NS>
struct Bars {
    static constexpr int KFULL = 0, VFULL = NS, EMPTY = 2 * NS, SFULL = 3 * NS, PFULL = SFULL + 2,
                         OFULL = PFULL + 2, QFULL = OFULL + 2, QEMPTY = QFULL + 2, DONE = QEMPTY + 2;
};

struct Ctl {
    volatile int* abort;
    int* err;
};

// Bounded wait: spins on try_wait; gives up after kWaitLimitNs or once the
// CTA's abort flag is set.  A timeout raises PKV_DEVERR_TIMEOUT and the flag.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const Ctl& c) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63) == 0) {
            if (*c.abort) return false;
            if (globaltimer_ns() - t0 > kWaitLimitNs) {
                raise_error(c.err, PKV_DEVERR_TIMEOUT);
                *c.abort = 1;
                return false;
            }
        }
    }
}

__device__ __forceinline__ bool bar_red_or(int id, int n, bool v) {
    uint32_t r;
    asm volatile(
        "{\n.reg .pred p, q;\nsetp.ne.u32 q, %1, 0;\nbar.red.or.pred p, %2, %3, q;\nselp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}

// Iterates the pieces of a CTA's unit range (every role walks it the same way).
struct PieceIter {
    Cursor cur;
    int u, u1, Hkv;
    int g, S0, S1, pg0, npg;
    __device__ void load(const AttnParams& p) {
        g = (u - cur.Ub) / cur.nb;
        S0 = cur.Ub + g * cur.nb;
        S1 = S0 + cur.nb;
        const int pe = min(u1, S1);
        pg0 = u - S0;
        npg = pe - u;
    }
    __device__ bool valid() const { return u < u1; }
    __device__ void advance(const AttnParams& p) {
        u += npg;
        if (u < u1 && u == cur.Ub + cur.nb * Hkv) cursor_next(p, cur);
        if (u < u1) load(p);
    }
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

template <int D, int NPAD, bool SPLIT, int NS>
__global__ void __launch_bounds__(kThreads, 1) attn_tc_kernel(const AttnParams p) {
    using K = Cfg<D, NPAD, SPLIT, NS>;
    using B = Bars<NS>;
    constexpr int RMAX = K::RMAX;
    extern __shared__ uint8_t smem_raw[];
    __shared__ int scratch[kThreads / 32 + 1];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    const uint32_t sb = smem_u32(smem);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    Cursor cur0;
    int u0, u1, W, P;
    if (!plan_locate<kThreads>(p, blockIdx.x, gridDim.x, scratch, &cur0, &u0, &u1, &W, &P)) return;
    const int cta = blockIdx.x;

    auto bar = [&](int i) -> uint32_t { return sb + K::OFF_BAR + 8 * i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + K::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + K::OFF_MISC + 4);
    volatile int* ticket_flag = reinterpret_cast<volatile int*>(smem + K::OFF_MISC + 8);
    volatile int* never = reinterpret_cast<volatile int*>(smem + K::OFF_MISC + 12);   // stays 0
    const Ctl ctl{abort_flag, p.err};
    const Ctl drain{never, p.err};      // bounded waits that ignore the abort flag

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(bar(B::KFULL + s), 1);
            mbar_init(bar(B::VFULL + s), 1);
            mbar_init(bar(B::EMPTY + s), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(B::SFULL + i), 1);
            mbar_init(bar(B::PFULL + i), kSoftThreads);
            mbar_init(bar(B::OFULL + i), 1);
            mbar_init(bar(B::QFULL + i), 1);
            mbar_init(bar(B::QEMPTY + i), 1);
        }
        mbar_init(bar(B::DONE), 1);
        *abort_flag = 0;
        *never = 0;
        mbar_fence_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), K::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int G = p.group, Hkv = p.num_kv_heads;

    PieceIter it;
    it.cur = cur0;
    it.u = u0;
    it.u1 = u1;
    it.Hkv = Hkv;
    it.load(p);

    if (warp == kProducerWarp) {
        // ------------------------------------------------------------ producer
        const uint64_t pol = policy_evict_first();
        int t = 0, j = 0;
        bool ok = true;
        while (ok && it.valid()) {
            const int qb = j & 1;
            if (j >= 2) {
                bool w = lane == 0 ? wait_bar(bar(B::QEMPTY + qb), ((j >> 1) - 1) & 1, ctl) : true;
                ok = __shfl_sync(0xffffffffu, w, 0);
                if (!ok) break;
            }
            // q rows of this (b, g) -> Q buffer in the K-major core-matrix layout
            const int R = G * it.cur.Q;
            uint8_t* qdst = smem + K::OFF_Q + qb * K::QBUF;
            for (int idx = lane; idx < NPAD * K::NCH; idx += 32) {
                const int r = idx / K::NCH, c = idx % K::NCH;
                uint4 v = make_uint4(0, 0, 0, 0);
                if (r < R) {
                    const int i = r / G, hl = r % G;
                    v = __ldg(reinterpret_cast<const uint4*>(
                        p.q + ((size_t)(it.cur.qoff + i) * p.num_q_heads + it.g * G + hl) * D + c * 8));
                }
                *reinterpret_cast<uint4*>(qdst + (r >> 3) * (K::NCH * 128) + c * 128 + (r & 7) * 16) = v;
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B::QFULL + qb));

            const int32_t* table = p.block_tables + (size_t)it.cur.b * p.max_blocks_per_seq;
            int ids = 0, ids_base = -1;
            for (int t0 = 0; t0 < it.npg; t0 += kTP, ++t) {
                const int np = min(kTP, it.npg - t0);
                const int st = t % NS;
                // block ids of this and the next 3 tiles, 8 per tile, one per lane
                if ((t0 >> 5) != ids_base) {
                    ids_base = t0 >> 5;
                    const int pi = (ids_base << 5) + lane;
                    ids = pi < it.npg ? table[it.pg0 + pi] : 0;
                }
                int blk = __shfl_sync(0xffffffffu, ids, ((t0 & 31) + (lane & 7)) & 31);
                if (t >= NS) {
                    bool w = lane == 0 ? wait_bar(bar(B::EMPTY + st), ((t / NS) - 1) & 1, ctl) : true;
                    ok = __shfl_sync(0xffffffffu, w, 0);
                    if (!ok) break;
                }
                if (lane == 0) {
                    mbar_arrive_expect_tx(bar(B::KFULL + st), np * K::PAGE);
                    mbar_arrive_expect_tx(bar(B::VFULL + st), np * K::PAGE);
                }
                __syncwarp();
                if (lane < np) {
                    if (blk < 0 || blk >= p.num_blocks) {
                        raise_error(p.err, PKV_DEVERR_BLOCK_ID);
                        blk = 0;
                    }
                    const size_t off = ((size_t)blk * Hkv + it.g) * K::PAGE;
                    bulk_g2s_hint(sb + K::OFF_K + st * K::TILE + lane * K::PAGE, p.k_cache + off, K::PAGE,
                                  bar(B::KFULL + st), pol);
                    bulk_g2s_hint(sb + K::OFF_V + st * (K::TILE + K::VSLACK) + lane * K::PAGE, p.v_cache + off,
                                  K::PAGE, bar(B::VFULL + st), pol);
                }
                __syncwarp();
            }
            ++j;
            it.advance(p);
        }
        // drain: the last fill of every stage has landed before the CTA exits
        if (lane == 0) {
            for (int tt = max(0, t - NS); tt < t; ++tt) {
                const int st = tt % NS;
                wait_bar(bar(B::KFULL + st), (tt / NS) & 1, drain);
                wait_bar(bar(B::VFULL + st), (tt / NS) & 1, drain);
            }
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idS = idesc_bf16_f32(128, NPAD, false, false);
            constexpr uint32_t idPV = idesc_bf16_f32(128, NPAD, true, true);
            int t = 0, j = 0;
            int pend = -1, pend_np = 0;
            bool ok = true;
            auto issue_pv = [&](int tt, int np) -> bool {
                const int st = tt % NS;
                if (!wait_bar(bar(B::VFULL + st), (tt / NS) & 1, ctl)) return false;
                if (!wait_bar(bar(B::PFULL + (tt & 1)), (tt >> 1) & 1, ctl)) return false;
                tc_fence_after();
                const uint32_t vbase = sb + K::OFF_V + st * (K::TILE + K::VSLACK);
                const uint32_t pbase = sb + K::OFF_P + (tt & 1) * K::PBUF;
                for (int pg = 0; pg < np; ++pg) {
                    const uint64_t a = smem_desc(vbase + pg * K::PAGE, K::NCH * 128, 128);
                    const uint64_t b = smem_desc(pbase + pg * 256, 128, 16 * 128);
                    mma_bf16(tmem + 2 * NPAD + (tt & 1) * NPAD, a, b, idPV, pg > 0);
                }
                mma_commit(bar(B::OFULL + (tt & 1)));
                mma_commit(bar(B::EMPTY + st));
                return true;
            };
            while (ok && it.valid()) {
                const int qb = j & 1;
                if (!(ok = wait_bar(bar(B::QFULL + qb), (j >> 1) & 1, ctl))) break;
                tc_fence_after();
                const uint32_t qbase = sb + K::OFF_Q + qb * K::QBUF;
                for (int t0 = 0; t0 < it.npg; t0 += kTP, ++t) {
                    const int np = min(kTP, it.npg - t0);
                    const int st = t % NS;
                    if (!(ok = wait_bar(bar(B::KFULL + st), (t / NS) & 1, ctl))) break;
                    tc_fence_after();
                    const uint32_t kbase = sb + K::OFF_K + st * K::TILE;
#pragma unroll
                    for (int k = 0; k < D / 16; ++k) {
                        const uint64_t a = smem_desc(kbase + k * 256, 128, K::NCH * 128);
                        const uint64_t b = smem_desc(qbase + k * 256, 128, K::NCH * 128);
                        mma_bf16(tmem + (t & 1) * NPAD, a, b, idS, k > 0);
                    }
                    mma_commit(bar(B::SFULL + (t & 1)));
                    if (t0 + kTP >= it.npg) mma_commit(bar(B::QEMPTY + qb));
                    if (pend >= 0 && !(ok = issue_pv(pend, pend_np))) break;
                    pend = t;
                    pend_np = np;
                }
                ++j;
                if (ok) it.advance(p);
            }
            if (ok && pend >= 0) issue_pv(pend, pend_np);
            mma_commit(bar(B::DONE));
            wait_bar(bar(B::DONE), 0, drain);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax / correction / epilogue
        const int tt = tid;                                   // token row of S^T, d row of O^T
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        float* red = reinterpret_cast<float*>(smem + K::OFF_RED);
        float* lred = reinterpret_cast<float*>(smem + K::OFF_LRED);
        int t = 0;
        bool aborted = false;
        float m_run[RMAX], l_part[RMAX], acc[RMAX], alpha_prev[RMAX];

        auto correct = [&](int tix) {
            bool w = wait_bar(bar(B::OFULL + (tix & 1)), (tix >> 1) & 1, ctl);
            (void)w;
            tc_fence_after();
            float o[NPAD];
#pragma unroll
            for (int c = 0; c < NPAD; c += 16) {
                float tmp[16];
                tmem_ld16(tmem + lane_base + 2 * NPAD + (tix & 1) * NPAD + c, tmp);
#pragma unroll
                for (int x = 0; x < 16; ++x) o[c + x] = tmp[x];
            }
#pragma unroll
            for (int r = 0; r < RMAX; ++r) {
                const float add = SPLIT ? (o[2 * r] + o[2 * r + 1]) : o[r];
                acc[r] = acc[r] * alpha_prev[r] + add;
            }
            tc_fence_before();
        };

        while (!aborted && it.valid()) {
            const int Q = it.cur.Q, R = G * Q, L = it.cur.L, lim0 = L - Q;
            const int st_b = it.cur.b;
#pragma unroll
            for (int r = 0; r < RMAX; ++r) {
                m_run[r] = -INFINITY;
                l_part[r] = 0.f;
                acc[r] = 0.f;
                alpha_prev[r] = 1.f;
            }
            const int ntile = (it.npg + kTP - 1) / kTP;
            for (int jt = 0; jt < ntile; ++jt, ++t) {
                const int np = min(kTP, it.npg - jt * kTP);
                const int st = t % NS;
                bool okw = wait_bar(bar(B::SFULL + (t & 1)), (t >> 1) & 1, ctl);
                tc_fence_after();
                float s[NPAD];
#pragma unroll
                for (int c = 0; c < NPAD; c += 16) {
                    float tmp[16];
                    tmem_ld16(tmem + lane_base + (t & 1) * NPAD + c, tmp);
#pragma unroll
                    for (int x = 0; x < 16; ++x) s[c + x] = tmp[x];
                }
                const int pgi = tt >> 4;
                const int pos = (it.pg0 + jt * kTP + pgi) * kBlock + (tt & 15);
                const bool tok_ok = pgi < np && pos < L;
                float x[RMAX];
#pragma unroll
                for (int r = 0; r < RMAX; ++r) {
                    const bool vis = r < R && tok_ok && pos <= lim0 + r / G;
                    x[r] = vis ? s[r] * p.scale_log2 : -INFINITY;
                }
                // tile max per row over the 128 tokens
                float* rd = red + (t & 1) * 4 * RMAX;
#pragma unroll
                for (int r = 0; r < RMAX; ++r) {
                    if (r < R) {
                        float mx = x[r];
#pragma unroll
                        for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                        if (lane == 0) rd[warp * RMAX + r] = mx;
                    }
                }
                if (bar_red_or(1, kSoftThreads, !okw || *abort_flag)) {
                    aborted = true;
                    break;
                }
                float alpha[RMAX], pr[RMAX];
#pragma unroll
                for (int r = 0; r < RMAX; ++r) {
                    if (r < R) {
                        const float tm = fmaxf(fmaxf(rd[r], rd[RMAX + r]), fmaxf(rd[2 * RMAX + r], rd[3 * RMAX + r]));
                        const float mn = fmaxf(m_run[r], tm);
                        alpha[r] = (m_run[r] == -INFINITY) ? 0.f : exp2f(m_run[r] - mn);
                        m_run[r] = mn;
                        pr[r] = (x[r] == -INFINITY) ? 0.f : exp2f(x[r] - mn);
                        l_part[r] = l_part[r] * alpha[r] + pr[r];
                    } else {
                        alpha[r] = 1.f;
                        pr[r] = 0.f;
                    }
                }
                // P^T row of this token: NPAD bf16 columns, MN-major core-matrix layout
                uint8_t* pdst = smem + K::OFF_P + (t & 1) * K::PBUF + tt * 16;
#pragma unroll
                for (int cc = 0; cc < NPAD / 8; ++cc) {
                    uint32_t w4[4];
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        float a, b;
                        if constexpr (SPLIT) {
                            const int r = cc * 4 + h;          // columns 2r (high) and 2r+1 (low)
                            const float hi = __bfloat162float(__float2bfloat16_rn(pr[r]));
                            a = hi;
                            b = pr[r] - hi;
                        } else {
                            a = pr[cc * 8 + 2 * h];
                            b = pr[cc * 8 + 2 * h + 1];
                        }
                        w4[h] = pack_bf16x2(a, b);
                    }
                    *reinterpret_cast<uint4*>(pdst + cc * (16 * 128)) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                }
                // unwritten tail slots of the sequence's last page: zero their V rows (they may hold NaN)
                if (pgi < np && pos >= L) {
                    wait_bar(bar(B::VFULL + st), (t / NS) & 1, ctl);
                    uint8_t* vrow = smem + K::OFF_V + st * (K::TILE + K::VSLACK) + pgi * K::PAGE +
                                    ((tt & 15) >> 3) * (K::NCH * 128) + (tt & 7) * 16;
#pragma unroll
                    for (int c = 0; c < K::NCH; ++c) *reinterpret_cast<uint4*>(vrow + c * 128) = make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(bar(B::PFULL + (t & 1)));
                if (jt > 0) correct(t - 1);
#pragma unroll
                for (int r = 0; r < RMAX; ++r) alpha_prev[r] = alpha[r];
            }
            if (aborted) break;
            correct(t - 1);

            // ---- epilogue of the piece: row sums, then output or partial
#pragma unroll
            for (int r = 0; r < RMAX; ++r) {
                if (r < R) {
                    float v = l_part[r];
#pragma unroll
                    for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                    if (lane == 0) lred[warp * RMAX + r] = v;
                }
            }
            named_bar_sync(1, kSoftThreads);
            float Lsum[RMAX];
#pragma unroll
            for (int r = 0; r < RMAX; ++r)
                Lsum[r] = (r < R) ? lred[r] + lred[RMAX + r] + lred[2 * RMAX + r] + lred[3 * RMAX + r] : 1.f;
            named_bar_sync(1, kSoftThreads);
            const bool complete = (it.S0 >= u0) && (it.S1 <= u1);
            if (complete) {
                if (tt < D) {
#pragma unroll
                    for (int r = 0; r < RMAX; ++r) {
                        if (r < R) {
                            const int i = r / G, hl = r % G;
                            p.out[((size_t)(it.cur.qoff + i) * p.num_q_heads + it.g * G + hl) * D + tt] =
                                __float2bfloat16_rn(acc[r] / Lsum[r]);
                        }
                    }
                }
            } else {
                float* slot = slot_ptr(p, cta, it.S0, u0);
#pragma unroll
                for (int r = 0; r < RMAX; ++r) {
                    if (r < R) {
                        if (tt == r) {
                            slot[r] = m_run[r];
                            slot[p.rows_pad + r] = Lsum[r];
                        }
                        if (tt < D) slot[2 * p.rows_pad + (size_t)r * D + tt] = acc[r];
                    }
                }
                __threadfence();
                named_bar_sync(1, kSoftThreads);
                if (tt == 0) {
                    const int need = owner_cta(it.S1 - 1, W, P) - owner_cta(it.S0, W, P) + 1;
                    const int old = atomicAdd(p.tickets + st_b * Hkv + it.g, 1);
                    const int last = (old == need - 1);
                    if (last) p.tickets[st_b * Hkv + it.g] = 0;
                    *ticket_flag = last;
                }
                named_bar_sync(1, kSoftThreads);
                if (*ticket_flag) {
                    __threadfence();
                    merge_segment<kSoftThreads>(p, it.cur, it.g, it.S0, it.S1, W, P, D);
                }
                named_bar_sync(1, kSoftThreads);
            }
            it.advance(p);
        }
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, K::TMEM_COLS);
    }
}

template <int D, int NPAD, bool SPLIT, int NS>
static cudaError_t launch_t(const AttnParams& p, int ncta, cudaStream_t st) {
    using K = Cfg<D, NPAD, SPLIT, NS>;
    auto kern = attn_tc_kernel<D, NPAD, SPLIT, NS>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, K::SMEM);
    if (e != cudaSuccess) return e;
    kern<<<ncta, kThreads, K::SMEM, st>>>(p);
    return cudaGetLastError();
}

}  // namespace tc

// bf16 cache, head_dim 64/128, R = G * max_q_len <= 32.
cudaError_t launch_attention_tc(const AttnParams& p, int head_dim, int ncta, cudaStream_t st) {
    const bool small = p.rows <= 8;
    if (head_dim == 128)
        return small ? tc::launch_t<128, 16, true, 3>(p, ncta, st) : tc::launch_t<128, 32, false, 3>(p, ncta, st);
    return small ? tc::launch_t<64, 16, true, 6>(p, ncta, st) : tc::launch_t<64, 32, false, 6>(p, ncta, st);
}

}  // namespace pkv
