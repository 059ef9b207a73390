// Paged chunked prefill: causal attention of long query windows (hundreds to
// thousands of new tokens per sequence) over the same paged cache, on the
// 5th-generation tensor cores (the lfm25-inference README's ragged/segmented
// prefill attention; the inferd backlog's chunked prefill).  Same result as
// pkv_paged_attention (the paged-KV equivalence: attention through the block
// table equals dense attention): query i of sequence b, query head h, sees
// positions 0 .. L_b - Q_b + i of kv-head h / G.
//
// A CTA owns 128 query rows of one kv-head: 128 / G consecutive query
// positions x the G heads of the group (row r = position r / G, head r % G),
// so every K/V page it streams serves all of them.  It walks 128-key tiles
// (8 pages) up to its rows' causal limit:
//   S[128 rows, 128 keys] = Q[128, D] . K_tile^T      (M=128, N=128, K-major A and B from shared memory)
//   softmax per row (one thread per row = TMEM lane, two reads of S: max, then P)
//   O[128 rows, D] += P_hi . V_tile + P_lo . V_tile   (M=128, N=D, A from TMEM, B MN-major in shared memory)
// S (two buffers), P and O live in TMEM.  P = 2^(s - m) is split into a bf16
// high part and the bf16 rounding of its remainder, so the weights keep ~16
// significant bits (one bf16 P misses the 2e-3 tolerance on rows that
// average a handful of keys); P_hi is written over the S columns already
// read, P_lo into its own columns.  The cache's page layout is already the
// canonical no-swizzle operand layout: K pages are K-major B operands, V pages
// MN-major B operands, so pages go HBM -> shared memory by 1-D bulk copies.
// O is rescaled in TMEM only when a row's maximum rises by more than 2^8
// (exp2 units).  Every mbarrier wait is bounded (the launch's wait limit).
//
// Roles: warps 0-3 softmax and epilogue (thread = row), warp 4 producer (block
// table, bulk copies), warp 5 MMA issuer (S of tile t, then P.V of tile t - 1;
// tcgen05.mma ops of one thread run in issue order, so S of tile t + 2 is
// written over P_hi of tile t only after P.V of tile t has read it).
#include "common.cuh"
#include "tc_ptx.cuh"

namespace pkv {
namespace prefill {

using namespace ptx;

constexpr int kRows = 128;                // query rows per CTA (MMA M)
constexpr int kTP = 8;                    // pages per key tile
constexpr int kKeys = kTP * kBlock;       // 128 keys per tile (MMA N of S)
constexpr int kThreads = 192;             // 4 softmax warps, producer, MMA issuer
constexpr int kProducer = 4, kMma = 5;
constexpr float kSlack = 8.f;             // rescale O only when a row's max rises by more than 2^8

template <int D>
struct Cfg {
    static constexpr int NCH = D / 8;                     // 16-byte chunks per row of D bf16
    static constexpr int PAGE = kBlock * D * 2;           // a bf16 page
    static constexpr int TILE = kTP * PAGE;
    static constexpr int NS = D == 128 ? 3 : 4;           // K and V ring depth (tiles)
    static constexpr int OFF_Q = 0;                       // Q [16 row groups][D/8][8][8]
    static constexpr int QBYTES = kRows * D * 2;
    static constexpr int OFF_K = OFF_Q + QBYTES;          // K ring
    static constexpr int OFF_V = OFF_K + NS * TILE;       // V ring
    static constexpr int OFF_BAR = OFF_V + NS * TILE;
    // barriers: KFULL[NS] VFULL[NS] KEMPTY[NS] VEMPTY[NS] SFULL[2] PFULL[2] PEMPTY[2] QFULL ODONE
    static constexpr int KFULL = 0, VFULL = NS, KEMPTY = 2 * NS, VEMPTY = 3 * NS, SFULL = 4 * NS,
                         PFULL = 4 * NS + 2, PEMPTY = 4 * NS + 4, QFULL = 4 * NS + 6, ODONE = 4 * NS + 7;
    static constexpr int NBAR = 4 * NS + 8;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;   // tmem address, abort flags, qoff
    static constexpr int SMEM = OFF_MISC + 16 + 128;      // (+ alignment slack)
    // TMEM columns: S / P_hi [2] x 128, O (D), P_lo [2] x 64
    static constexpr int COL_O = 2 * kKeys;
    static constexpr int COL_LO = COL_O + D;
    static constexpr int TMEM_COLS = 512;
    static_assert(COL_LO + 2 * (kKeys / 2) <= TMEM_COLS, "tensor memory budget");
    static_assert(SMEM <= 232448 - 1024, "shared memory budget");
};

struct Ctl {
    volatile int* abort;
    int* err;
    uint64_t limit;
};

__device__ __noinline__ bool wait_spin(uint32_t bar, uint32_t parity, volatile int* abort, int* err, uint64_t limit) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63) == 0) {
            if (*abort) return false;
            if (globaltimer_ns() - t0 > limit) {
                raise_error(err, PKV_DEVERR_TIMEOUT);
                *abort = 1;
                return false;
            }
        }
    }
}
__device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity, const Ctl& c) {
    if (mbar_try_wait(bar, parity)) return true;
    return wait_spin(bar, parity, c.abort, c.err, c.limit);
}

__device__ __forceinline__ float exp2_fast(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(const AttnParams p, int qblocks) {
    using K = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    const uint32_t sb = smem_u32(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    auto bar = [&](int i) -> uint32_t { return sb + K::OFF_BAR + 8 * i; };
    constexpr int NS = K::NS, KFULL = K::KFULL, VFULL = K::VFULL, KEMPTY = K::KEMPTY, VEMPTY = K::VEMPTY,
                  SFULL = K::SFULL, PFULL = K::PFULL, PEMPTY = K::PEMPTY, QFULL = K::QFULL, ODONE = K::ODONE;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + K::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + K::OFF_MISC + 4);
    int* s_qoff = reinterpret_cast<int*>(smem + K::OFF_MISC + 8);
    // abort flag of the drain waits at the end (set only when one of them runs out)
    volatile int* drain_flag = reinterpret_cast<volatile int*>(smem + K::OFF_MISC + 12);
    const Ctl ctl{abort_flag, p.err, p.wait_limit_ns};

    griddep_launch();
    griddep_wait();
    // this CTA: sequence b, kv-head g, query block qb of 128 / G positions (the
    // last blocks, which see the most keys, first)
    const int G = p.group, QP = kRows / G;
    const int qb = qblocks - 1 - (int)(blockIdx.x % qblocks), g = (blockIdx.x / qblocks) % p.num_kv_heads,
              b = blockIdx.x / (qblocks * p.num_kv_heads);
    const int L = p.context_lens[b], Q = p.q_lens[b];
    const int q0 = qb * QP;
    // uniform over the CTA: nothing to do (past the window, or invalid lengths: the first CTA reports those)
    const bool bad = Q > L || Q < 0 || Q > p.max_q_len || (L + kBlock - 1) / kBlock > p.max_blocks_per_seq;
    if (bad && q0 == 0 && g == 0 && tid == 0 && Q != 0) raise_error(p.err, PKV_DEVERR_LENGTH);
    if (bad || q0 >= Q) return;
    const int nq = min(QP, Q - q0);                       // query positions of this CTA
    const int lim_max = L - Q + q0 + nq - 1;              // last key any of its rows sees
    const int T = lim_max / kKeys + 1;                    // key tiles
    const int nb = (L + kBlock - 1) / kBlock;             // pages of the sequence

    if (tid == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(bar(KFULL + i), 1);
            mbar_init(bar(VFULL + i), 1);
            mbar_init(bar(KEMPTY + i), 1);
            mbar_init(bar(VEMPTY + i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(SFULL + i), 1);
            mbar_init(bar(PFULL + i), kRows);
            mbar_init(bar(PEMPTY + i), 1);
        }
        mbar_init(bar(QFULL), kRows);
        mbar_init(bar(ODONE), 1);
        *abort_flag = 0;
        *drain_flag = 0;
        mbar_fence_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), K::TMEM_COLS);
        tmem_relinquish();
        // first q row of sequence b
        int s = 0;
        for (int i = lane; i < b; i += 32) s += max(p.q_lens[i], 0);
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == 0) *s_qoff = s;
    }
    tc_fence_before();
    cta_bar_sync();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int qoff = *s_qoff;

    if (warp < 4) {
        // ------------------------------------------------ softmax / epilogue: thread r = row r
        const int r = tid, qi = r / G, hl = r - qi * G;
        const bool row_ok = qi < nq;
        const int qpos = L - Q + q0 + qi;                 // this row's query position (last key it sees)
        const uint32_t lbase = (uint32_t)(warp * 32) << 16;
        // q row -> Q tile (K-major core matrices), zeros for rows past the window
        {
            const uint4* src = reinterpret_cast<const uint4*>(
                p.q + ((size_t)(qoff + q0 + qi) * p.num_q_heads + g * G + hl) * D);
            uint8_t* dst = smem + K::OFF_Q + (r >> 3) * (K::NCH * 128) + (r & 7) * 16;
#pragma unroll 4
            for (int c = 0; c < K::NCH; ++c)
                *reinterpret_cast<uint4*>(dst + c * 128) = row_ok ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
            fence_proxy_async_smem();
            mbar_arrive(bar(QFULL));
        }
        // keys 0 .. lim are visible to this row (lim <= L - 1; -1: a row past the window)
        const int lim = row_ok ? qpos : -1;
        // every wait and every TMEM access of the loop is warp-uniform (tcgen05.ld/st are .aligned)
        auto wait_all = [&](uint32_t bb, uint32_t parity) { return __all_sync(0xffffffffu, wait(bb, parity, ctl)); };
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int t = 0; t < T && ok; ++t) {
            const int s = t & 1;
            if (!(ok = wait_all(bar(SFULL + s), (t >> 1) & 1))) break;
            tc_fence_after();
            const uint32_t scol = tmem + lbase + s * kKeys;
            const int rem = lim - t * kKeys;               // column c is visible iff c <= rem
            // pass 1: the tile's maximum for this row
            float tmax = -INFINITY;
#pragma unroll
            for (int c = 0; c < kKeys; c += 16) {
                float v[16];
                tmem_ld16(scol + c, v);
#pragma unroll
                for (int x = 0; x < 16; ++x) tmax = fmaxf(tmax, c + x <= rem ? v[x] * p.scale_log2 : -INFINITY);
            }
            // a new maximum more than 2^8 above the running one: rescale l and O
            const bool grow = tmax > m + kSlack || (m == -INFINITY && tmax > -INFINITY);
            const float alpha = !grow ? 1.f : (m == -INFINITY ? 0.f : exp2_fast(m - tmax));
            if (t > 0 && __any_sync(0xffffffffu, grow && m != -INFINITY)) {
                // O *= alpha (1 for the warp's other rows), once the previous tile's P.V has landed
                if (!(ok = wait_all(bar(PEMPTY + ((t - 1) & 1)), ((t - 1) >> 1) & 1))) break;
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < D; c += 16) {
                    float o[16];
                    tmem_ld16(tmem + lbase + K::COL_O + c, o);
#pragma unroll
                    for (int x = 0; x < 16; ++x) o[x] *= alpha;
                    tmem_st16(tmem + lbase + K::COL_O + c, o);
                }
            }
            l *= alpha;
            if (grow) m = tmax;
            // pass 2: P = 2^(s - m) -> P_hi over the S columns already read, P_lo in its own
            // columns (column j / 2 of a part holds keys j, j + 1; the even key in the low half).
            // Their previous contents were read by the P.V of tile t - 2, which completed
            // before S of tile t (issued after it) signalled SFULL.
            const uint32_t phi = tmem + lbase + s * kKeys, plo = tmem + lbase + K::COL_LO + s * (kKeys / 2);
#pragma unroll
            for (int c = 0; c < kKeys; c += 16) {
                float v[16];
                tmem_ld16(scol + c, v);
                uint32_t wh[8], wl[8];
#pragma unroll
                for (int x = 0; x < 16; x += 2) {
                    const float p0 = c + x <= rem ? exp2_fast(v[x] * p.scale_log2 - m) : 0.f;
                    const float p1 = c + x + 1 <= rem ? exp2_fast(v[x + 1] * p.scale_log2 - m) : 0.f;
                    l += p0 + p1;
                    const __nv_bfloat162 h = __floats2bfloat162_rn(p0, p1);
                    const __nv_bfloat162 lo = __floats2bfloat162_rn(p0 - __low2float(h), p1 - __high2float(h));
                    wh[x >> 1] = *reinterpret_cast<const uint32_t*>(&h);
                    wl[x >> 1] = *reinterpret_cast<const uint32_t*>(&lo);
                }
                tmem_st8(phi + (c >> 1), wh);
                tmem_st8(plo + (c >> 1), wl);
            }
            tmem_wait_st();
            tc_fence_before();
            // the last page's unwritten slots: zero their V rows (they may hold NaN)
            if (t == T - 1 && nb * kBlock > L && (nb - 1) / kTP == t) {
                if (!(ok = wait_all(bar(VFULL + t % NS), (t / NS) & 1))) break;
                const int tail = nb * kBlock - L, pg = (nb - 1) % kTP;
                for (int i = r; i < tail * K::NCH; i += kRows) {
                    const int key = kBlock - tail + i / K::NCH, c = i % K::NCH;
                    uint8_t* vrow = smem + K::OFF_V + (t % NS) * K::TILE + pg * K::PAGE +
                                    (key >> 3) * (K::NCH * 128) + c * 128 + (key & 7) * 16;
                    *reinterpret_cast<uint4*>(vrow) = make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();
            }
            mbar_arrive(bar(PFULL + s));
        }
        // epilogue: O / l -> out
        if (ok && wait_all(bar(ODONE), 0)) {
            tc_fence_after();
            __nv_bfloat16* dst = p.out + ((size_t)(qoff + q0 + qi) * p.num_q_heads + g * G + hl) * D;
#pragma unroll
            for (int c = 0; c < D; c += 16) {
                float o[16];
                tmem_ld16(tmem + lbase + K::COL_O + c, o);
                if (row_ok) {
                    uint32_t w[8];
#pragma unroll
                    for (int x = 0; x < 16; x += 2) {
                        __nv_bfloat162 pr = __floats2bfloat162_rn(__fdividef(o[x], l), __fdividef(o[x + 1], l));
                        w[x >> 1] = *reinterpret_cast<uint32_t*>(&pr);
                    }
                    *reinterpret_cast<uint4*>(dst + c) = make_uint4(w[0], w[1], w[2], w[3]);
                    *reinterpret_cast<uint4*>(dst + c + 8) = make_uint4(w[4], w[5], w[6], w[7]);
                }
            }
        }
    } else if (warp == kProducer) {
        // ------------------------------------------------ producer: K and V pages of each tile
        const int32_t* table = p.block_tables + (size_t)b * p.max_blocks_per_seq;
        int kc = 0;
        bool ok = true;
        if (p.hold != nullptr) {
            // (tests of the timeout path only) wait, bounded, for a flag that nothing sets
            bool w = true;
            if (lane == 0) {
                const uint64_t h0 = globaltimer_ns();
                while (*reinterpret_cast<const volatile int*>(p.hold) == 0) {
                    if (*abort_flag || globaltimer_ns() - h0 > p.wait_limit_ns) {
                        if (!*abort_flag) raise_error(p.err, PKV_DEVERR_TIMEOUT);
                        *abort_flag = 1;
                        w = false;
                        break;
                    }
                    __nanosleep(256);
                }
            }
            ok = __shfl_sync(0xffffffffu, w, 0);
        }
        for (int t = 0; t < T && ok; ++t) {
            const int s = t % NS, p0 = t * kTP, np = min(kTP, nb - p0);
            const int sl = lane & 7, kv = lane >> 3;      // lanes 0-7 copy K pages, 8-15 V pages
            int blk = (kv < 2 && sl < np) ? __ldg(table + p0 + sl) : 0;
            if (kv < 2 && sl < np && (blk < 0 || blk >= p.num_blocks)) {
                if (kv == 0) raise_error(p.err, PKV_DEVERR_BLOCK_ID);
                blk = 0;
            }
            bool w = true;
            if (t >= NS) {
                if (lane == 0) w = wait(bar(KEMPTY + s), ((t - NS) / NS) & 1, ctl);
                if (lane == 8) w = wait(bar(VEMPTY + s), ((t - NS) / NS) & 1, ctl);
            }
            if (!(ok = __all_sync(0xffffffffu, w))) break;
            if (lane == 0) mbar_arrive_expect_tx(bar(KFULL + s), np * K::PAGE);
            if (lane == 8) mbar_arrive_expect_tx(bar(VFULL + s), np * K::PAGE);
            __syncwarp();
            if (kv < 2 && sl < np) {
                const size_t off = ((size_t)blk * p.cache_kv_heads + g) * K::PAGE;
                // (default cache policy: every query block of the sequence reads these pages, from L2)
                bulk_g2s(sb + (kv ? K::OFF_V : K::OFF_K) + s * K::TILE + sl * K::PAGE,
                         (kv ? p.v_cache : p.k_cache) + off, K::PAGE, bar((kv ? VFULL : KFULL) + s));
            }
            ++kc;
        }
        // drain: the copies in flight land before the CTA exits
        if (lane == 0) {
            const Ctl drain{drain_flag, p.err, p.wait_limit_ns};
            for (int t = max(0, kc - NS); t < kc; ++t) {
                wait(bar(KFULL + t % NS), (t / NS) & 1, drain);
                wait(bar(VFULL + t % NS), (t / NS) & 1, drain);
            }
        }
        __syncwarp();
    } else if (warp == kMma) {
        // ------------------------------------------------ MMA issuer: S of tile t, then P.V of tile t - 1
        if (lane == 0) {
            constexpr uint32_t idS = idesc_bf16_f32(kRows, kKeys, false, false);
            constexpr uint32_t idPV = idesc_bf16_f32(kRows, D, false, true);
            const uint32_t qbase = sb + K::OFF_Q;
            bool ok = wait(bar(QFULL), 0, ctl);
            auto pv = [&](int u) -> bool {
                const int su = u & 1, vs = u % NS, np = min(kTP, nb - u * kTP);
                if (!wait(bar(PFULL + su), (u >> 1) & 1, ctl)) return false;
                if (!wait(bar(VFULL + vs), (u / NS) & 1, ctl)) return false;
                tc_fence_after();
                const uint32_t vbase = sb + K::OFF_V + vs * K::TILE;
                const uint32_t ahi = tmem + su * kKeys, alo = tmem + K::COL_LO + su * (kKeys / 2);
                for (int pg = 0; pg < np; ++pg) {       // 16 keys per MMA: one page, 8 TMEM columns of P
                    const uint64_t bv = smem_desc(vbase + pg * K::PAGE, K::NCH * 128, 128);
                    mma_bf16_tmem_a(tmem + K::COL_O, ahi + pg * 8, bv, idPV, (u > 0 || pg > 0) ? 1u : 0u);
                    mma_bf16_tmem_a(tmem + K::COL_O, alo + pg * 8, bv, idPV, 1u);
                }
                mma_commit(bar(PEMPTY + su));
                mma_commit(bar(VEMPTY + vs));
                return true;
            };
            for (int t = 0; t < T && ok; ++t) {
                const int s = t & 1, ks = t % NS;
                if (!(ok = wait(bar(KFULL + ks), (t / NS) & 1, ctl))) break;
                tc_fence_after();
                const uint32_t kbase = sb + K::OFF_K + ks * K::TILE;
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint64_t a = smem_desc(qbase + k * 256, 128, K::NCH * 128);
                    const uint64_t bk = smem_desc(kbase + k * 256, 128, K::NCH * 128);
                    mma_bf16(tmem + s * kKeys, a, bk, idS, k > 0 ? 1u : 0u);
                }
                mma_commit(bar(SFULL + s));
                mma_commit(bar(KEMPTY + ks));
                if (t >= 1) ok = pv(t - 1);
            }
            if (ok) ok = pv(T - 1);
            mma_commit(bar(ODONE));
            // every MMA issued has completed before TMEM is freed
            const Ctl drain{drain_flag, p.err, p.wait_limit_ns};
            wait(bar(ODONE), 0, drain);
        }
        __syncwarp();
    }

    // teardown: every role arrives from its own code path (non-.aligned barrier)
    tc_fence_before();
    cta_bar_sync();
    if (warp == 0) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, K::TMEM_COLS);
    }
}

}  // namespace prefill

cudaError_t launch_prefill(const AttnParams& p, int head_dim, cudaStream_t st) {
    const int qblocks = (p.max_q_len * p.group + prefill::kRows - 1) / prefill::kRows;
    const int64_t grid = (int64_t)p.num_seqs * p.num_kv_heads * qblocks;
    if (grid < 1 || grid > 0x7fffffff) return cudaErrorInvalidValue;
    static std::atomic<uint64_t> set64{0}, set128{0};
    if (head_dim == 128)
        return launch_pdl_bigsmem(set128, prefill::prefill_kernel<128>, dim3((unsigned)grid), dim3(prefill::kThreads),
                                  (size_t)prefill::Cfg<128>::SMEM, st, p, qblocks);
    return launch_pdl_bigsmem(set64, prefill::prefill_kernel<64>, dim3((unsigned)grid), dim3(prefill::kThreads),
                              (size_t)prefill::Cfg<64>::SMEM, st, p, qblocks);
}

}  // namespace pkv
