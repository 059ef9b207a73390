// Paged chunked prefill: causal attention of long query windows (hundreds to
// thousands of new tokens per sequence) over the same paged cache, on the
// 5th-generation tensor cores (the lfm25-inference README's ragged/segmented
// prefill attention; the inferd backlog's chunked prefill).  Same result as
// pkv_paged_attention (the paged-KV equivalence: attention through the block
// table equals dense attention): query i of sequence b, query head h, sees
// positions 0 .. L_b - Q_b + i of kv-head h / G.
//
// A work item is 256 query rows of one kv-head -- 256 / G consecutive query
// positions x the G heads of the group (row r = position r / G, head r % G)
// -- held as two 128-row tiles, so every K/V page a CTA streams serves 256
// rows.  The CTAs are persistent (one per SM) and take items heavy first in
// serpentine rounds.  An item walks 128-key tiles (8 pages) up to its rows'
// causal limit; per key tile t and row tile i:
//   S_i[128 rows, 128 keys] = Q_i . K_t^T     (M=128, N=128, K-major A and B in shared memory)
//   softmax per row (one thread per row = TMEM lane), one pass against the
//     row's running reference maximum
//   O_i[128 rows, D] += P_i . V_t             (M=128, N=D, fp16 A from TMEM, fp16 B MN-major in shared memory)
// S, P and O live in TMEM (S/P_0, S/P_1: 128 columns each; O_0, O_1: D each).
// P = 2^(s - m) is written as fp16 pairs over the S columns already read
// (fp16 keeps 11 significant bits; bf16 P misses the 2e-3 tolerance on rows
// that average a handful of keys), and V is turned from bf16 into fp16 in
// shared memory once per tile, since both operands of one MMA have the same
// type.  The cache's page layout is already the canonical no-swizzle operand
// layout: K pages are K-major B operands, V pages MN-major B operands, so
// pages go HBM -> shared memory by 1-D bulk copies.  O is rescaled in TMEM
// only when a row's maximum rises by more than 2^8 (exp2 units).
//
// Roles (384 threads): warps 0-3 softmax of row tile 0, warps 4-7 of row
// tile 1 (thread = row; they also run the epilogue, and row tile 0 converts
// V), warp 8 the K producer and warp 9 the V producer (block table, bulk
// copies into their own rings), warps 10 and 11 the MMA issuers of row tiles
// 0 and 1.  Issuer i runs, per tile,
//   PV_i(t, first 64 keys) once their P is written | PV_i(t, rest) | S_i(t + 1)
// so one row tile's softmax runs while the tensor core works for the other,
// and the first half of P.V overlaps the softmax of the second.
// tcgen05.mma ops of one thread run in issue order: S_i(t + 1) overwrites P_i
// only after PV_i(t) has read it, and when S_i(t + 1) signals, PV_i(t) has
// completed, so the softmax may rescale O_i without another wait.  Every
// mbarrier wait is bounded (the launch's wait limit).
#include <algorithm>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace pkv {
namespace prefill {

using namespace ptx;

constexpr int kRows = 128;                // rows per row tile (MMA M)
constexpr int kCtaRows = 2 * kRows;       // rows per CTA
constexpr int kTP = 8;                    // pages per key tile
constexpr int kKeys = kTP * kBlock;       // 128 keys per tile (MMA N of S)
constexpr int kThreads = 384;             // 8 softmax warps, K producer, V producer, 2 MMA issuers
constexpr int kProdK = 8, kProdV = 9, kMma = 10;   // MMA issuers: warps 10 and 11
constexpr float kSlack = 8.f;             // rescale O only when a row's max rises by more than 2^8

template <int D>
struct Cfg {
    static constexpr int NCH = D / 8;                     // 16-byte chunks per row of D bf16
    static constexpr int PAGE = kBlock * D * 2;           // a bf16 page
    static constexpr int TILE = kTP * PAGE;
    static constexpr int NSK = D == 128 ? 2 : 4;          // K ring depth (tiles)
    static constexpr int NSV = D == 128 ? 3 : 4;          // V ring depth: V(t + 1) lands during tile t
    static constexpr int QBYTES = kRows * D * 2;          // one row tile of Q: [16 row groups][D/8][8][8]
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + 2 * QBYTES;      // K ring
    static constexpr int OFF_V = OFF_K + NSK * TILE;      // V ring
    static constexpr int OFF_BAR = OFF_V + NSV * TILE;
    // barriers: KFULL[NSK] KEMPTY[NSK] VFULL[NSV] VEMPTY[NSV] VREADY[NSV] SFULL[2] PFA[2] PFB[2] PVA[2]
    // QFULL ODONE[2] OFREE[2] DRAIN  (PFA / PFB: P of a tile's first / last 64 keys written; PVA: the
    // P.V of its first 64 keys done)
    static constexpr int KFULL = 0, KEMPTY = NSK, VFULL = 2 * NSK, VEMPTY = 2 * NSK + NSV,
                         VREADY = 2 * NSK + 2 * NSV, SFULL = 2 * NSK + 3 * NSV, PFA = SFULL + 2, PFB = SFULL + 4,
                         PVA = SFULL + 6, QFULL = SFULL + 8, ODONE = SFULL + 9, OFREE = SFULL + 11,
                         DRAIN = SFULL + 13;
    static constexpr int NBAR = SFULL + 14;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;   // tmem address, abort flags, qoff
    static constexpr int SMEM = OFF_MISC + 16 + 128;      // (+ alignment slack)
    // TMEM columns: S/P_0, S/P_1 (128 each), O_0, O_1 (D each)
    static constexpr int COL_O = 2 * kKeys;
    static constexpr int TMEM_COLS = 512;
    static_assert(COL_O + 2 * D <= TMEM_COLS, "tensor memory budget");
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

// Two fp32 lanes in one 64-bit register (the sm_100 family's packed fp32 arithmetic).
__device__ __forceinline__ uint64_t f2pack(uint32_t a, uint32_t b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};\n" : "=l"(r) : "r"(a), "r"(b));
    return r;
}
__device__ __forceinline__ void f2unpack(uint64_t r, float& a, float& b) {
    asm("mov.b64 {%0, %1}, %2;\n" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t f2fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;\n" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t f2add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;\n" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// One work item: 256 / G query positions (query block qb) of sequence b and kv-head g.  Items are
// numbered heavy first -- the last query blocks, which see the most keys, of every (sequence,
// kv-head), then the ones before -- and the persistent CTAs deal them out in serpentine rounds
// (round k gives item k * grid + c to CTA c on even rounds, k * grid + grid - 1 - c on odd ones),
// which keeps the CTAs' loads close when the items' costs fall off.
struct Item {
    int b, g, q0, nq, L, Q, T, nb;
    bool two;           // row tile 1 holds rows of the window
};
__device__ __forceinline__ bool item_at(const AttnParams& p, int j, int qblocks, Item& it) {
    const int bg = p.num_seqs * p.num_kv_heads;
    const int qb = qblocks - 1 - j / bg;
    it.b = (j % bg) / p.num_kv_heads;
    it.g = (j % bg) % p.num_kv_heads;
    it.L = p.context_lens[it.b];
    it.Q = p.q_lens[it.b];
    it.q0 = qb * (kCtaRows / p.group);
    const bool bad = it.Q > it.L || it.Q < 0 || it.Q > p.max_q_len ||
                     (it.L + kBlock - 1) / kBlock > p.max_blocks_per_seq;
    if (bad || it.q0 >= it.Q) return false;
    it.nq = min(kCtaRows / p.group, it.Q - it.q0);
    it.two = it.nq * p.group > kRows;
    it.T = (it.L - it.Q + it.q0 + it.nq - 1) / kKeys + 1;
    it.nb = (it.L + kBlock - 1) / kBlock;
    return true;
}
// This CTA's next item after its round k (k = -1: the first); k advances to the item's round.
// Returns the item's number, or `total` when none is left.
__device__ __forceinline__ int next_item(const AttnParams& p, int& k, int total, int qblocks, Item& it) {
    const int grid = gridDim.x, c = blockIdx.x;
    for (++k; (int64_t)k * grid < total; ++k) {
        const int j = k * grid + ((k & 1) ? grid - 1 - c : c);
        if (j < total && item_at(p, j, qblocks, it)) return j;
    }
    return total;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(const AttnParams p, int qblocks) {
    using K = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    const uint32_t sb = smem_u32(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    auto bar = [&](int i) -> uint32_t { return sb + K::OFF_BAR + 8 * i; };
    constexpr int NSK = K::NSK, NSV = K::NSV, KFULL = K::KFULL, VFULL = K::VFULL, KEMPTY = K::KEMPTY,
                  VEMPTY = K::VEMPTY, VREADY = K::VREADY,
                  SFULL = K::SFULL, PFA = K::PFA, PFB = K::PFB, PVA = K::PVA, QFULL = K::QFULL, ODONE = K::ODONE,
                  OFREE = K::OFREE, DRAIN = K::DRAIN;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + K::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + K::OFF_MISC + 4);
    // abort flag of the drain waits at the end (set only when one of them runs out)
    volatile int* drain_flag = reinterpret_cast<volatile int*>(smem + K::OFF_MISC + 12);
    const Ctl ctl{abort_flag, p.err, p.wait_limit_ns};

    griddep_launch();
    griddep_wait();
    const int G = p.group;
    const int total = p.num_seqs * p.num_kv_heads * qblocks;
    // invalid lengths are reported once, by the CTA that owns the sequence's first item of kv-head 0
    if (tid == 0)
        for (int k = 0; (int64_t)k * gridDim.x < total; ++k) {
            const int j = k * gridDim.x + ((k & 1) ? gridDim.x - 1 - blockIdx.x : blockIdx.x);
            const int bg = p.num_seqs * p.num_kv_heads, b = (j % bg) / p.num_kv_heads;
            if (j < total && j / bg == qblocks - 1 && (j % bg) % p.num_kv_heads == 0) {
                const int L = p.context_lens[b], Q = p.q_lens[b];
                if (Q != 0 && (Q > L || Q < 0 || Q > p.max_q_len || (L + kBlock - 1) / kBlock > p.max_blocks_per_seq))
                    raise_error(p.err, PKV_DEVERR_LENGTH);
            }
        }
    Item first;
    int k0 = -1;
    const int j0 = next_item(p, k0, total, qblocks, first);
    if (j0 >= total) return;                              // (uniform over the CTA)

    if (tid == 0) {
        for (int i = 0; i < NSK; ++i) {
            mbar_init(bar(KFULL + i), 1);
            mbar_init(bar(KEMPTY + i), 2);                // both MMA issuers release every K tile
        }
        for (int i = 0; i < NSV; ++i) {
            mbar_init(bar(VFULL + i), 1);
            mbar_init(bar(VEMPTY + i), 2);
            mbar_init(bar(VREADY + i), kRows);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(SFULL + i), 1);
            mbar_init(bar(PFA + i), kRows);
            mbar_init(bar(PFB + i), kRows);
            mbar_init(bar(PVA + i), 1);
            mbar_init(bar(ODONE + i), 1);
            mbar_init(bar(OFREE + i), kRows);
        }
        mbar_init(bar(QFULL), kCtaRows);
        mbar_init(bar(DRAIN), 2);
        *abort_flag = 0;
        *drain_flag = 0;
        mbar_fence_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), K::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    cta_bar_sync();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp < 8) {
        // ------------------------------------------------ softmax / epilogue: row tile i, thread r = row r
        const int i = warp >> 2, r = tid & (kRows - 1);
        const int R = i * kRows + r, qi = R / G, hl = R - qi * G;   // row R: query position qi of the item, head hl
        const uint32_t lbase = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t scol = tmem + lbase + i * kKeys;   // S_i / P_i
        const uint32_t ocol = tmem + lbase + K::COL_O + i * D;
        // every wait and every TMEM access of the loop is warp-uniform (tcgen05.ld/st are .aligned)
        auto wait_all = [&](uint32_t bb, uint32_t parity) { return __all_sync(0xffffffffu, wait(bb, parity, ctl)); };
        int nb = 0, valid_last = kBlock;                   // the current item's pages, its last page's tokens
        const float sc = p.scale_log2;
        int rem_c = 0;                                     // this tile: column c is visible iff c <= rem_c
        // P of 32 keys (S values rr, columns c .. c + 31) -> 16 columns of fp16 pairs (the even key
        // in the low half) at column c / 2, over S columns already read.  MASK: keys past this
        // row's limit weigh 0.  Adds P to ls[].
        auto emit = [&](const uint32_t (&rr)[32], int c, float mref, bool mask, float (&ls)[2]) {
            uint32_t w[16];
#pragma unroll
            for (int k = 0; k < 32; k += 2) {
                float p0 = exp2_fast(fmaf(__uint_as_float(rr[k]), sc, -mref));
                float p1 = exp2_fast(fmaf(__uint_as_float(rr[k + 1]), sc, -mref));
                if (mask) {
                    p0 = c + k <= rem_c ? p0 : 0.f;
                    p1 = c + k + 1 <= rem_c ? p1 : 0.f;
                }
                ls[0] += p0;
                ls[1] += p1;
                const __half2 h = __floats2half2_rn(p0, p1);
                w[k >> 1] = *reinterpret_cast<const uint32_t*>(&h);
            }
            tmem_st16u(scol + (c >> 1), w);
        };
        // O_i *= alpha (1 for rows that keep their reference); warp-uniform
        auto rescale_o = [&](float alpha) {
#pragma unroll 1
            for (int c = 0; c < D; c += 32) {
                float o[32];
                tmem_ld32(ocol + c, o);
                uint32_t w[16];
#pragma unroll
                for (int x = 0; x < 16; ++x) w[x] = __float_as_uint(o[x] * alpha);
                tmem_st16u(ocol + c, w);
#pragma unroll
                for (int x = 0; x < 16; ++x) w[x] = __float_as_uint(o[16 + x] * alpha);
                tmem_st16u(ocol + c + 16, w);
            }
            tmem_wait_st();
        };
        // m: this row's reference maximum (exp2 units); pend: a maximum that the last tile raised
        // by more than the slack, applied to l and O when the next tile starts (PV_i of the last
        // tile has completed by then).  In one pass, P = 2^(s - m) is kept below 2^kBig (inside
        // the fp16 range): a chunk that would exceed it first raises m by a whole number k of
        // octaves, and the P this tile already holds, O and l are scaled by 2^-k (exact but for
        // fp16 subnormals: weights below 2^-14 of the new maximum).
        constexpr float kBig = 15.f;
        float m = -INFINITY, l = 0.f, pend = -INFINITY;
        // (sent_a: this tile's first 64 keys' P has been signalled; its P.V then also reads them, so
        // once that P.V has completed, O holds them and only the P written since is rescaled)
        bool sent_a = false;
        int cur_tile = 0;                                  // this row tile's tile number (PVA phase)
        auto raise_ref = [&](float target, int c, uint64_t& acc) {
            const float inc = target > m + kBig ? fminf(ceilf(target - m), 254.f) : 0.f;
            const int k = (int)inc;
            const float alpha = k < 127 ? __uint_as_float((uint32_t)(127 - k) << 23) : 0.f;
            int c0 = 0;
            if (sent_a) {
                wait_all(bar(PVA + i), cur_tile & 1);
                tc_fence_after();
                c0 = kKeys / 4;                            // (P of the first 64 keys: 32 columns)
            }
#pragma unroll 1
            for (int cc = c0; cc < c / 2; cc += 16) {         // the P columns written so far
                float o[16];
                tmem_ld16(scol + cc, o);
                uint32_t w[16];
#pragma unroll
                for (int x = 0; x < 16; ++x) {
                    const uint32_t u = __float_as_uint(o[x]);
                    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&u));
                    const __half2 h = __floats2half2_rn(f.x * alpha, f.y * alpha);
                    w[x] = *reinterpret_cast<const uint32_t*>(&h);
                }
                tmem_st16u(scol + cc, w);
            }
            rescale_o(alpha);
            l *= alpha;
            float a0, a1;
            f2unpack(acc, a0, a1);
            acc = f2pack(__float_as_uint(a0 * alpha), __float_as_uint(a1 * alpha));
            m += inc;
        };
        // P of 32 keys, two keys per packed fp32 operation (MASK: keys past this row's limit weigh
        // 0); unless FORCE, nothing is stored (false) when the chunk's sum of P reaches 2^kBig (or
        // is NaN): P >= 0, so no P reaches it otherwise.  Adds the chunk's P to acc.
        auto emit_fast = [&](const uint32_t (&rr)[32], int c, uint64_t& acc, bool force, bool mask) -> bool {
            const uint64_t sc2 = f2pack(__float_as_uint(sc), __float_as_uint(sc));
            const uint64_t nm2 = f2pack(__float_as_uint(-m), __float_as_uint(-m));
            uint64_t ca = 0;                               // (+0, +0)
            uint32_t w[16];
#pragma unroll
            for (int k = 0; k < 32; k += 2) {
                float x0, x1;
                f2unpack(f2fma(f2pack(rr[k], rr[k + 1]), sc2, nm2), x0, x1);
                float p0 = exp2_fast(x0), p1 = exp2_fast(x1);
                if (mask) {
                    p0 = c + k <= rem_c ? p0 : 0.f;
                    p1 = c + k + 1 <= rem_c ? p1 : 0.f;
                }
                ca = f2add(ca, f2pack(__float_as_uint(p0), __float_as_uint(p1)));
                const __half2 h = __floats2half2_rn(p0, p1);
                w[k >> 1] = *reinterpret_cast<const uint32_t*>(&h);
            }
            if (!force) {
                float c0, c1;
                f2unpack(ca, c0, c1);
                if (__any_sync(0xffffffffu, !(c0 + c1 < 32768.f))) return false;
            }
            acc = f2add(acc, ca);
            tmem_st16u(scol + (c >> 1), w);
            return true;
        };
        auto chunk = [&](const uint32_t (&rr)[32], int c, uint64_t& acc, bool mask) {
            if (emit_fast(rr, c, acc, false, mask)) return;
            // (rare) a logit more than 2^kBig above the reference: raise it first
            float c0 = -INFINITY, c1 = -INFINITY;
#pragma unroll
            for (int x = 0; x < 32; x += 2) {
                c0 = fmaxf(c0, !mask || c + x <= rem_c ? __uint_as_float(rr[x]) : -INFINITY);
                c1 = fmaxf(c1, !mask || c + x + 1 <= rem_c ? __uint_as_float(rr[x + 1]) : -INFINITY);
            }
            raise_ref(fmaxf(c0, c1) * sc, c, acc);
            emit_fast(rr, c, acc, true, mask);              // (P <= 1 now, but for NaN logits)
        };
        // one pass over a tile once the row's reference is known, loads of the next 32 columns in
        // flight while the previous 32 are turned into P; returns the tile's sum of P
        auto fast_pass = [&](bool mask) -> float {
            uint64_t acc = 0;
            uint32_t ra[32], rb[32];
            tmem_ld32_async(scol, ra);
            tmem_wait_ld_into(ra);
#pragma unroll 1
            for (int c = 0; c < kKeys; c += 64) {
                tmem_ld32_async(scol + c + 32, rb);
                chunk(ra, c, acc, mask);
                tmem_wait_ld_into(rb);
                if (c + 64 < kKeys) tmem_ld32_async(scol + c + 64, ra);
                chunk(rb, c + 32, acc, mask);
                if (c == 0) {
                    // the first 64 keys' P is complete: their P.V may run while the rest is computed
                    tmem_wait_st();
                    tc_fence_before();
                    mbar_arrive(bar(PFA + i));
                    sent_a = true;
                }
                if (c + 64 < kKeys) tmem_wait_ld_into(ra);
            }
            float a0, a1;
            f2unpack(acc, a0, a1);
            return a0 + a1;
        };
        // V(t), once landed, from bf16 to fp16 in place for the fp16 P.V products, by row tile 0:
        // V(t + 1) right after it signals P_0(t), while its next S is computed, so that its P_0(t + 1)
        // signal also says V(t + 1) is ready; VREADY tells row tile 1's MMA issuer.
        // Exact for |v| < 65536
        // (bf16 values carry 8 significant bits; below 2^-14 they become fp16 subnormals, off by
        // less than 2^-25); a finite |v| >= 65536 sets PKV_DEVERR_RANGE.  The last page's
        // unwritten slots become 0 (they may hold NaN).
        constexpr int CPP = K::PAGE / 16;                  // 16-byte chunks per page
        uint32_t vmaxbits = 0;                             // largest |bf16| bit patterns seen (two halves)
        // tile t of the current item, the CTA's V tile number gt (ring slot and phase)
        auto convert_v = [&](int gt, int t) -> bool {
            const int s = gt % NSV, np = min(kTP, nb - t * kTP), lastpg = nb - 1 - t * kTP;
            if (!wait_all(bar(VFULL + s), (gt / NSV) & 1)) return false;
            uint4* base = reinterpret_cast<uint4*>(smem + K::OFF_V + s * K::TILE);
            for (int pg = 0; pg < np; ++pg) {
                uint4* pgp = base + pg * CPP;
                const bool last = pg == lastpg && valid_last < kBlock;
#pragma unroll
                for (int e = r; e < CPP; e += kRows) {
                    uint4 v = pgp[e];
                    // chunk e of a page: token group e / (8 NCH), token (e % 8) of the group
                    if (last && (e / (K::NCH * 8)) * 8 + (e & 7) >= valid_last) {
                        v = make_uint4(0, 0, 0, 0);
                    } else {
                        uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            vmaxbits = __vmaxu2(vmaxbits, w[j] & 0x7fff7fffu);
                            const __half2 h = __floats2half2_rn(__uint_as_float(w[j] << 16),
                                                                __uint_as_float(w[j] & 0xffff0000u));
                            w[j] = *reinterpret_cast<const uint32_t*>(&h);
                        }
                    }
                    pgp[e] = v;
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(bar(VREADY + s));
            return true;
        };
        // The CTA's items in order.  Per item: its q rows -> Q_i, (row tile 0) V of its first tile
        // converted, the softmax of each key tile (row tile 0 converting the next tile's V after
        // signalling P), and the epilogue, during which the next item's q rows are already loaded.
        int scnt = 0, ocnt = 0, gv = 0;                    // this row tile's S tiles and items; V tiles
        bool ok = true;
        Item it = first;
        int j = j0, kr = k0;
        auto qsum = [&](int b) {                           // first q row of sequence b
            int sum = 0;
            for (int x = lane; x < b; x += 32) sum += max(p.q_lens[x], 0);
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
            return sum;
        };
        int qoff = qsum(it.b);
        auto q_row = [&](const Item& x, int xoff) {       // this row's q in the item (row 0 past the window)
            return reinterpret_cast<const uint4*>(
                p.q + ((size_t)(xoff + x.q0 + (qi < x.nq ? qi : 0)) * p.num_q_heads + x.g * G + hl) * D);
        };
        while (ok && j < total) {
            // q rows -> Q tile i (K-major core matrices), zeros for rows past the window.  This warp's
            // rows of the Q_i area held its staged output of the last item: the bulk copies have read it.
            {
                const bool rok = qi < it.nq;
                const uint4* src = q_row(it, qoff);
                uint8_t* dst = smem + K::OFF_Q + i * K::QBYTES + (r >> 3) * (K::NCH * 128) + (r & 7) * 16;
                uint4 qv[K::NCH];                          // all loads in flight at once
#pragma unroll
                for (int c = 0; c < K::NCH; ++c) qv[c] = rok ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
#pragma unroll
                for (int c = 0; c < K::NCH; ++c) *reinterpret_cast<uint4*>(dst + c * 128) = qv[c];
                fence_proxy_async_smem();
                mbar_arrive(bar(QFULL));
            }
            const bool act = i == 0 || it.two;
            const int T = it.T;
            nb = it.nb;
            valid_last = it.L - (it.nb - 1) * kBlock;
            const bool row_ok = qi < it.nq;
            // keys 0 .. lim are visible to this row (lim <= L - 1; -1: a row past the window)
            const int lim = row_ok ? it.L - it.Q + it.q0 + qi : -1;
            if (i == 0) ok = convert_v(gv, 0);
            m = -INFINITY;
            l = 0.f;
            pend = -INFINITY;
            for (int t = 0; act && t < T && ok; ++t) {
                if (!(ok = wait_all(bar(SFULL + i), scnt & 1))) break;
                tc_fence_after();
                rem_c = lim - t * kKeys;
                cur_tile = scnt;
                sent_a = false;
                if (__any_sync(0xffffffffu, pend > m + kSlack)) {
                    const bool up = pend > m + kSlack;
                    const float alpha = up ? exp2_fast(m - pend) : 1.f;
                    rescale_o(alpha);
                    l *= alpha;
                    if (up) m = pend;
                }
                pend = -INFINITY;
                if (__all_sync(0xffffffffu, m > -INFINITY) && sc > 0.f) {
                    // reference known: one pass (masked on the causal diagonal).  A tile sum of P of
                    // 2^e or more (e >= kSlack; it bounds the largest P) moves the reference up by
                    // e + 1 octaves at the next tile.
                    const float ts = __all_sync(0xffffffffu, rem_c >= kKeys - 1) ? fast_pass(false) : fast_pass(true);
                    l += ts;
                    if (ts >= 256.f && ts < INFINITY) pend = m + (float)((int)(__float_as_uint(ts) >> 23) - 127 + 1);
                } else {
                    // two passes (a warp's first tile with keys, rows past the window): the tile's
                    // maximum over the visible keys first, then P
                    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll 1
                    for (int c = 0; c < kKeys; c += 32) {
                        float v[32];
                        tmem_ld32(scol + c, v);
#pragma unroll
                        for (int x = 0; x < 32; ++x)
                            mx[x & 1] = fmaxf(mx[x & 1], c + x <= rem_c ? v[x] * sc : -INFINITY);
                    }
                    const float tmax = fmaxf(mx[0], mx[1]);
                    const bool grow = tmax > m + kSlack || (m == -INFINITY && tmax > -INFINITY);
                    const float alpha = !grow ? 1.f : (m == -INFINITY ? 0.f : exp2_fast(m - tmax));
                    if (t > 0 && __any_sync(0xffffffffu, grow && m != -INFINITY)) rescale_o(alpha);
                    l *= alpha;
                    if (grow) m = tmax;
                    // rows with nothing visible yet keep m = -inf: every P of theirs is masked to 0
                    const float mref = m == -INFINITY ? 0.f : m;
                    float ls[2] = {0.f, 0.f};
#pragma unroll 1
                    for (int c = 0; c < kKeys; c += 32) {
                        uint32_t rr[32];
                        tmem_ld32_async(scol + c, rr);
                        tmem_wait_ld_into(rr);
                        emit(rr, c, mref, true, ls);
                    }
                    l += ls[0] + ls[1];
                }
                tmem_wait_st();
                tc_fence_before();
                if (!sent_a) mbar_arrive(bar(PFA + i));
                mbar_arrive(bar(PFB + i));
                ++scnt;
                if (i == 0 && t + 1 < T && !(ok = convert_v(gv + t + 1, t + 1))) break;
            }
            if (!ok) break;
            gv += T;
            // the next item: its q rows are brought to L2 while this item's epilogue runs
            const Item cur = it;
            const int cur_off = qoff;
            j = next_item(p, kr, total, qblocks, it);
            if (j < total) {
                qoff = qsum(it.b);
                if (qi < it.nq) {
                    const char* a = reinterpret_cast<const char*>(q_row(it, qoff));
#pragma unroll
                    for (int c = 0; c < D * 2; c += 128) asm volatile("prefetch.global.L2 [%0];\n" ::"l"(a + c));
                }
            }
            // epilogue: O_i / l -> bf16 rows [row][D] in the Q_i area (free: every S of the item has
            // completed when ODONE_i signals), then one bulk copy per run of a warp's rows that share
            // a query position (its consecutive heads, contiguous in out)
            if (act) {
                if (!(ok = wait_all(bar(ODONE + i), ocnt & 1))) break;
                tc_fence_after();
                uint8_t* stg = smem + K::OFF_Q + R * (D * 2);
                const float inv = 1.f / l;
#pragma unroll 1
                for (int c = 0; c < D; c += 32) {
                    float o[32];
                    tmem_ld32(ocol + c, o);
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        uint32_t w[4];
#pragma unroll
                        for (int x = 0; x < 4; ++x) {
                            __nv_bfloat162 pr = __floats2bfloat162_rn(o[h * 8 + 2 * x] * inv, o[h * 8 + 2 * x + 1] * inv);
                            w[x] = *reinterpret_cast<uint32_t*>(&pr);
                        }
                        *reinterpret_cast<uint4*>(stg + (c + h * 8) * 2) = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
                tc_fence_before();
                mbar_arrive(bar(OFREE + i));               // O_i read: the next item's PV may overwrite it
                ++ocnt;
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    const int R0 = R;                      // (lane 0: the warp's first row)
                    for (int Rr = R0; Rr < R0 + 32;) {
                        const int qq = Rr / G, hh = Rr - qq * G, n = min(G - hh, R0 + 32 - Rr);
                        if (qq < cur.nq)
                            bulk_s2g(p.out + ((size_t)(cur_off + cur.q0 + qq) * p.num_q_heads + cur.g * G + hh) * D,
                                     sb + K::OFF_Q + Rr * (D * 2), (uint32_t)(n * D * 2));
                        Rr += n;
                    }
                    bulk_commit_group();
                    bulk_wait_read();                      // the staging rows are free again
                }
                __syncwarp();
            }
        }
        if (lane == 0) bulk_wait_all();                    // every output row written
        {
            const uint32_t lo = vmaxbits & 0xffffu, hi = vmaxbits >> 16;
            if ((lo >= 0x4780u && lo < 0x7f80u) || (hi >= 0x4780u && hi < 0x7f80u)) raise_error(p.err, PKV_DEVERR_RANGE);
        }
    } else if (warp == kProdK || warp == kProdV) {
        // ------------------------------------------------ producers: K pages (warp 8) and V pages (warp 9)
        // of each tile, each through its own ring (one lane per page)
        const bool isv = warp == kProdV;
        const int NSR = isv ? NSV : NSK, FULL = isv ? VFULL : KFULL, EMPTY = isv ? VEMPTY : KEMPTY;
        const uint32_t ring = sb + (isv ? K::OFF_V : K::OFF_K);
        const uint8_t* src = isv ? p.v_cache : p.k_cache;
        int kc = 0;                                       // tiles issued (over the CTA's items)
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
        Item it = first;
        int kr = k0;
        for (int j = j0; j < total && ok; j = next_item(p, kr, total, qblocks, it)) {
            const int32_t* table = p.block_tables + (size_t)it.b * p.max_blocks_per_seq;
            for (int t = 0; t < it.T && ok; ++t) {
                const int s = kc % NSR, p0 = t * kTP, np = min(kTP, it.nb - p0);
                int blk = lane < np ? __ldg(table + p0 + lane) : 0;
                if (lane < np && (blk < 0 || blk >= p.num_blocks)) {
                    if (!isv) raise_error(p.err, PKV_DEVERR_BLOCK_ID);
                    blk = 0;
                }
                bool w = true;
                if (kc >= NSR && lane == 0) w = wait(bar(EMPTY + s), ((kc - NSR) / NSR) & 1, ctl);
                if (!(ok = __shfl_sync(0xffffffffu, w, 0))) break;
                if (lane == 0) mbar_arrive_expect_tx(bar(FULL + s), np * K::PAGE);
                __syncwarp();
                // (default cache policy: every query block of the sequence reads these pages, from L2)
                if (lane < np)
                    bulk_g2s(ring + s * K::TILE + lane * K::PAGE,
                             src + ((size_t)blk * p.cache_kv_heads + it.g) * K::PAGE, K::PAGE, bar(FULL + s));
                ++kc;
            }
        }
        // drain: the copies in flight land before the CTA exits
        if (lane == 0) {
            const Ctl drain{drain_flag, p.err, p.wait_limit_ns};
            for (int t = max(0, kc - NSR); t < kc; ++t) wait(bar(FULL + t % NSR), (t / NSR) & 1, drain);
        }
        __syncwarp();
    } else if (warp == kMma || warp == kMma + 1) {
        // ------------------------------------------------ MMA issuers, one per row tile i (warp 10: i = 0,
        // warp 11: i = 1): PV_i(t) once P_i(t) is written, then S_i(t + 1) once K(t + 1) has landed.
        // Each row tile's S, P and O sit in its own TMEM columns and one thread's tcgen05.mma ops
        // run in issue order; while one issuer waits for its P, the other keeps the tensor core fed.
        const int i = warp - kMma;
        if (lane == 0) {
            constexpr uint32_t idS = idesc_bf16_f32(kRows, kKeys, false, false);
            constexpr uint32_t idPV = idesc_f16_f32(kRows, D, false, true);
            const uint32_t qbase = sb + K::OFF_Q + i * K::QBYTES, sfull = tmem + i * kKeys;
            int gk = 0, gvt = 0;                          // the CTA's K and V tiles so far (ring slots, phases)
            int pcnt = 0, ocnt = 0, n = 0;                // this row tile's P tiles and items; the CTA's items
            Item it = first;
            auto issue_s = [&](int t) {
                const int kt = gk + t;
                const uint32_t kbase = sb + K::OFF_K + (kt % NSK) * K::TILE;
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint64_t a = smem_desc(qbase + k * 256, 128, K::NCH * 128);
                    const uint64_t bk = smem_desc(kbase + k * 256, 128, K::NCH * 128);
                    mma_bf16(sfull, a, bk, idS, k > 0 ? 1u : 0u);
                }
                mma_commit(bar(SFULL + i));
                mma_commit(bar(KEMPTY + kt % NSK));       // (K(t) is free once both row tiles' S(t) ran)
            };
            // PV_i(t) over pages [pa, pz) of the tile: one page (16 keys = 8 columns of fp16 P_i pairs)
            // per MMA
            auto issue_pv = [&](int t, int pa, int pz) {
                const int vt = gvt + t;
                const uint32_t vbase = sb + K::OFF_V + (vt % NSV) * K::TILE;
                const uint32_t o = tmem + K::COL_O + i * D;
                for (int pg = pa; pg < pz; ++pg) {
                    const uint64_t bv = smem_desc(vbase + pg * K::PAGE, K::NCH * 128, 128);
                    mma_bf16_tmem_a(o, sfull + pg * 8, bv, idPV, (t > 0 || pg > 0) ? 1u : 0u);
                }
            };
            bool ok = true;
            int kr = k0;
            for (int j = j0; j < total && ok; j = next_item(p, kr, total, qblocks, it), ++n) {
                const int T = it.T;
                if (!(ok = wait(bar(QFULL), n & 1, ctl))) break;
                if (i == 0 || it.two) {
                    if (!(ok = wait(bar(KFULL + gk % NSK), (gk / NSK) & 1, ctl))) break;
                    tc_fence_after();
                    issue_s(0);
                    for (int t = 0; t < T && ok; ++t) {
                        // row tile 0 converts V(t) (before it signals P_0(t)): row tile 1 waits for it
                        if (i == 1 && !(ok = wait(bar(VREADY + (gvt + t) % NSV), ((gvt + t) / NSV) & 1, ctl))) break;
                        // P.V of the first 64 keys as soon as their P is written, of the rest after
                        const int np = min(kTP, it.nb - t * kTP);
                        if (!(ok = wait(bar(PFA + i), pcnt & 1, ctl))) break;
                        // the first PV of an item starts O_i afresh: the last item's epilogue has read it
                        if (t == 0 && ocnt > 0 && !(ok = wait(bar(OFREE + i), (ocnt - 1) & 1, ctl))) break;
                        tc_fence_after();
                        issue_pv(t, 0, min(np, kTP / 2));
                        mma_commit(bar(PVA + i));
                        if (!(ok = wait(bar(PFB + i), pcnt & 1, ctl))) break;
                        ++pcnt;
                        tc_fence_after();
                        issue_pv(t, kTP / 2, np);
                        mma_commit(bar(VEMPTY + (gvt + t) % NSV));
                        if (t + 1 < T) {
                            const int kt = gk + t + 1;
                            if (!(ok = wait(bar(KFULL + kt % NSK), (kt / NSK) & 1, ctl))) break;
                            tc_fence_after();
                            issue_s(t + 1);
                        } else {
                            mma_commit(bar(ODONE + i));
                        }
                    }
                    ++ocnt;
                } else {
                    // row tile 1 has no rows in this item: release its share of every K and V slot,
                    // each once that slot's tile has landed (so the arrival counts for that tile)
                    for (int t = 0; t < T && ok; ++t) {
                        const int kt = gk + t, vt = gvt + t;
                        if (!(ok = wait(bar(KFULL + kt % NSK), (kt / NSK) & 1, ctl))) break;
                        mma_commit(bar(KEMPTY + kt % NSK));
                        if (!(ok = wait(bar(VFULL + vt % NSV), (vt / NSV) & 1, ctl))) break;
                        mma_commit(bar(VEMPTY + vt % NSV));
                    }
                }
                gk += T;
                gvt += T;
            }
            mma_commit(bar(DRAIN));
            // every MMA issued has completed before TMEM is freed
            const Ctl drain{drain_flag, p.err, p.wait_limit_ns};
            wait(bar(DRAIN), 0, drain);
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

cudaError_t launch_prefill(const AttnParams& p, int head_dim, int num_sms, cudaStream_t st) {
    // persistent: one CTA per SM (at most one per work item), taking items round-robin
    const int qblocks = (int)(((int64_t)p.max_q_len * p.group + prefill::kCtaRows - 1) / prefill::kCtaRows);
    const int64_t items = (int64_t)p.num_seqs * p.num_kv_heads * qblocks;
    if (items < 1 || items > 0x7fffffff || num_sms < 1) return cudaErrorInvalidValue;
    const unsigned grid = (unsigned)std::min<int64_t>(items, num_sms);
    static std::atomic<uint64_t> set64{0}, set128{0};
    if (head_dim == 128)
        return launch_pdl_bigsmem(set128, prefill::prefill_kernel<128>, dim3(grid), dim3(prefill::kThreads),
                                  (size_t)prefill::Cfg<128>::SMEM, st, p, qblocks);
    return launch_pdl_bigsmem(set64, prefill::prefill_kernel<64>, dim3(grid), dim3(prefill::kThreads),
                              (size_t)prefill::Cfg<64>::SMEM, st, p, qblocks);
}

}  // namespace pkv
