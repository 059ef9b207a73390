// Paged decode / verify attention on the 5th-generation tensor cores
// (tcgen05 MMA, accumulators in TMEM, pages staged by 1-D bulk copies).
//
// Computes what attn_simt.cu computes (the paged GQA/XQA attention of the
// lfm25-inference README, equal to dense attention per the inferd
// equivalence gate): for every sequence b and query row (i, query head h),
//   out = softmax_j(scale * q . k_j) v_j,  j <= L - Q + i,  kv-head h / G.
//
// Columns.  A segment is (sequence b, group of HG kv-heads).  Its query rows
// sit on the MMA's N side ("swap AB"): column n = hh * R + r for kv-head
// hh of the group and row r = i * G + hl of that head's GQA group, R = G * Q,
// NCOL = HG * R <= 8 (P split into a bf16 high and low part on adjacent
// columns, N = 16) or <= 32 (N = 32; P's low parts in a second ring, and
// instances whose softmax handles only the first 20 or 24 columns).  A
// 128-token tile holds 8 (page,
// kv-head) units in page-major order; each token row only sees the columns of
// its own kv-head.
//
// Per tile:
//   S^T[128 tok, N] = K_tile[128 tok, D] . Q^T[D, N]        (M=128, K-major A and B)
//   softmax on S^T rows (one thread per token, TMEM lane = token)
//   O^T[128 d, N]  += V_tile^T[d, 128 tok] . P^T[128 tok, N] (M=128, MN-major A and B)
// K and V pages sit in separate rings: a K slot is refilled as soon as its
// S^T MMA has run, a V slot once its P.V MMA has.
//
// O^T stays in TMEM for the whole piece; pieces alternate between two
// accumulators, so a piece's epilogue overlaps the next piece's tiles.  The
// softmax reference max of a column is only raised (and O^T rescaled in TMEM)
// when a logit exceeds it by more than 2^8, so most tiles need neither a max
// reduction nor a rescale.
//
// The cache's page layout (16-byte chunks, core matrices of 8 tokens x 16
// bytes, see pagedkv.h) is the tensor core's no-swizzle canonical layout: K
// pages are K-major A operands and V pages MN-major A operands as copied, so
// a page goes HBM -> shared memory in one bulk copy and is never touched by
// the CUDA cores (except zeroing the unwritten tail rows of a sequence's last
// page, which may hold NaN).
//
// FP8 (e4m3) caches, NCOL <= 8 (N = 16) or, at head_dim 128, <= 16 (N = 32):
// the K pages stay e4m3 and S^T runs on kind::f8f6f4 MMAs against the q
// rows, each scaled by a power of two and split exactly into two e4m3 terms
// (columns n and NCOL-max + n, added in the softmax with the page's k scale);
// the V pages land in the upper half of a bf16 operand slot and the softmax
// warpgroup widens them in place after writing each tile's P; P carries the
// page's v scale.  Page scales reach a ring in shared memory by cp.async.
//
// Work partition: the balanced unit partition of common.cuh, one persistent
// CTA per SM (for wide and FP8 segments, cut by weight with a fixed charge
// per segment).  A CTA takes its last piece first and then walks its range
// from the start, so
// both pieces of every segment cut between two CTAs finish early and their
// merge overlaps the rest of the work.
//
// Split segments: a split piece's epilogue stores its partial (m, l, acc) and
// hands it to the merge warp, which reads the segment's ticket: when every
// other piece is already published it merges at once; otherwise it publishes
// the partial (fence, ticket increment) and merges if its ticket was the last.
//
// Warp roles: warps 0-3 softmax and O rescale (each warp its TMEM lane
// quarter), warp 4 producer (bulk copies, q staging, one piece ahead on q and
// the block table), warp 5 the S^T issuer, warp 6 the merge warp, warp 7 the
// P.V issuer (the two issuers block on their own barriers, so a P.V never
// waits behind the next tiles' S^T), and warps 8-11, the epilogue warpgroup:
// piece epilogues run there, off the softmax's path (the bf16 wide instances
// of more than 20 columns, whose softmax needs the registers of a 256-thread
// block, run them in the softmax warps, after the next piece's first tile).  Every mbarrier wait is bounded (2 s); a timeout sets
// PKV_DEVERR_TIMEOUT and an abort flag, all roles wind down, in-flight copies
// are drained and TMEM is freed before the CTA exits.
#include "common.cuh"
#include "tc_ptx.cuh"

namespace pkv {
namespace tc {

using namespace ptx;

constexpr int kTP = 8;                        // units (pages of one kv-head) per tile
constexpr int kTileTok = kTP * kBlock;        // 128 token rows = MMA M
constexpr int kSoftThreads = 128;             // one warpgroup (the 128 TMEM lanes)
constexpr int kMaxSmem = 232448;
constexpr int NSB = 4;                        // S^T / P ring depth (tiles the MMA may run ahead)
// warps 0-3 softmax; 4 producer, 5 S^T issuer, 6 merge, 7 P.V issuer; with
// EWG, 8-11 the epilogue warpgroup.  Named barriers: 1 softmax, 2 epilogue.
constexpr int kProducerWarp = 4, kMmaWarp = 5, kMergeWarp = 6, kPvWarp = 7, kEpiWarp0 = 8;
constexpr int kBarSoft = 1, kBarEpi = 2;
template <bool EWG>
__host__ __device__ constexpr int threads_of() { return EWG ? 384 : 256; }
constexpr int kSeqTab = 256;                  // sequences the shared-memory table holds

// Online-softmax reference slack (powers of two), see the header comment.
constexpr float kRescaleSlack = 8.f;
// Units charged per segment in the weighted CTA cut of narrow FP8 segments
// (wide: 24); measured best of 4-40 on the long FP8 batch
constexpr int kNarrowCharge = 16;
// ... and of wide segments whose epilogue runs in the epilogue warpgroup (with it in the
// softmax warps: 24)
constexpr int kWideEwgCharge = 12;

template <int D, int NPAD, bool SPLIT, int NSK, int NSV, bool EWG, bool FP8>
struct Cfg {
    // logical columns: SPLIT, P's high and low parts on adjacent columns; FP8, S^T holds each q row
    // as two e4m3 terms on columns n and RMAX + n
    static constexpr int RMAX = (SPLIT || FP8) ? NPAD / 2 : NPAD;
    // MMA N: NPAD rounded up to 16 (a wide kernel with NPAD = 20 or 24 computes 32 columns, and
    // its softmax and epilogue touch only the first NPAD: P columns from the next multiple of 8
    // on are never written and only reach O columns that are never read)
    static constexpr int NM = (NPAD + 15) / 16 * 16;
    static constexpr int PAGE = kBlock * D * 2;         // a page as bf16 MMA operand
    static constexpr int PAGE8 = kBlock * D;            // an FP8 cache page
    static constexpr int NSC = 16;                      // scale ring: tiles the producer may lead by, bounded
    static constexpr int NCH = D / 8;                   // 16-byte chunks per token row
    static constexpr int TILE = kTP * PAGE;
    static constexpr int VSLACK = D == 64 ? 1024 : 0;   // M=128 PV on D=64 reads 1 KiB past a page
    // FP8: K tiles stay e4m3 (the S MMA takes them as they are); a V slot's
    // e4m3 pages land in its upper half and are widened to bf16 in place
    static constexpr int KSLOT = FP8 ? kTP * PAGE8 : TILE;
    static constexpr int OFF_K = 0;                     // + st * KSLOT
    static constexpr int OFF_V = NSK * KSLOT;           // + st * (TILE + VSLACK)
    static constexpr int OFF_LAND = TILE - kTP * PAGE8;
    // FP8 scale ring: float [NSC][32]: k scales [8], v scales [8], column factors [RMAX <= 16]
    static constexpr int OFF_SC = OFF_V + NSV * (TILE + VSLACK);
    static constexpr int OFF_Q = OFF_SC + (FP8 ? NSC * 32 * 4 : 0);
    static constexpr int QBUF = NM * D * 2;
    static constexpr int OFF_P = OFF_Q + 2 * QBUF;
    static constexpr int PBUF = NM * kTileTok * 2;
    // wide segments (no high/low columns) keep P's low parts in a second ring
    static constexpr int OFF_PLO = OFF_P + NSB * PBUF;
    static constexpr int OFF_RED = OFF_PLO + (SPLIT ? 0 : NSB * PBUF);  // float [8 slots][RMAX]
    static_assert(NSB * PBUF >= 384 * 16, "the P ring holds the planning scratch (int4 per sequence)");
    static constexpr int OFF_LRED = OFF_RED + 8 * RMAX * 4;            // float [2][4 warps][RMAX]
    static constexpr int OFF_EM = OFF_LRED + 2 * 4 * RMAX * 4;         // float [2][RMAX]
    static constexpr int OFF_PD = OFF_EM + 2 * RMAX * 4;               // int [2][8]: piece descriptors
    static constexpr int OFF_BAR = OFF_PD + 2 * 8 * 4;
    static constexpr int NBAR = 2 * NSK + 2 * NSV + 3 * NSB + 18 + (FP8 ? NSV + NSC : 0);   // the barriers of Bars
    static constexpr int OFF_MISC = (OFF_BAR + NBAR * 8 + 15) / 16 * 16;  // tmem addr, abort, zero, gather state
    static constexpr int OFF_MQ = OFF_MISC + 16;         // merge tasks: int [4][8]
    static constexpr int OFF_VOTE = OFF_MQ + 128;        // int [2][4]: the softmax warps' votes (tile parity)
    static constexpr int OFF_SEQ = OFF_VOTE + 32;        // int4 [SEQTAB]: per-sequence (L, Q, Ub, qoff)
    // pre-merged earlier pieces of the CTA's last segment: M[RMAX], den[RMAX], num[RMAX][D]
    static constexpr int SEQTAB = FP8 ? kSeqTab / 2 : kSeqTab;   // sequences the table holds
    static constexpr int OFF_GATHER = OFF_SEQ + SEQTAB * 16;
    static constexpr int GATHER = SPLIT ? RMAX * (D + 2) * 4 : 0;
    // the weighted CTA boundaries (int [TABMAX + 1])
    static constexpr int TABMAX = 160;
    static constexpr int OFF_BND = (OFF_GATHER + GATHER + 15) / 16 * 16;
    static constexpr bool PTAB = (FP8 || !SPLIT) && OFF_BND + (TABMAX + 1) * 4 + 128 <= kMaxSmem - 512;
    static constexpr int SMEM_USED = (PTAB ? OFF_BND + (TABMAX + 1) * 4 : OFF_GATHER + GATHER) + 128;  // + slack
    // One CTA per SM either way: take the whole per-block budget, so every
    // operand read the descriptors can form stays inside the allocation.
    static constexpr int SMEM = kMaxSmem - 512;         // (static shared memory: < 300 bytes)
    static constexpr int COL_S = 0;                      // S^T buffers: NSB x NM columns
    // O^T accumulators: [piece parity][kv-head of the segment] x NM columns.
    // Each kv-head of a segment accumulates into its own: a P.V MMA of one
    // head's page also multiplies the zero P entries of the other heads'
    // columns, and 0 x NaN (a NaN stored in the page's V) must not reach them.
    static constexpr int HGMAX = SPLIT ? 4 : 2;          // kv-heads per segment
    static constexpr int COL_O = NSB * NM;
    static constexpr int NCOLS = NSB * NM + 2 * HGMAX * NM;
    static constexpr int TMEM_COLS = NCOLS <= 64 ? 64 : NCOLS <= 128 ? 128 : 256;
    static_assert(NCOLS <= 256, "TMEM budget");
    static_assert(OFF_BAR % 8 == 0 && OFF_SEQ % 16 == 0 && OFF_RED % 16 == 0, "shared memory alignment");
    static_assert(SMEM_USED <= SMEM, "shared memory budget");
};

template <int NSK, int NSV, bool FP8>
struct Bars {
    static constexpr int KFULL = 0, KEMPTY = NSK, VFULL = 2 * NSK, VEMPTY = 2 * NSK + NSV,
                         SFULL = 2 * NSK + 2 * NSV, PFULL = SFULL + NSB, PEMPTY = PFULL + NSB,
                         QFULL = PEMPTY + NSB, QEMPTY = QFULL + 2, DONE = QEMPTY + 2, MQFULL = DONE + 2,
                         ODONE = MQFULL + 4,      // [2]: last P.V of a piece of that parity done
                         PREADY = ODONE + 2,      // [2]: a piece of that parity handed to the epilogue
                         OFREE = PREADY + 2,      // [2]: its epilogue has read O^T, lred and emref
                         VOTE = OFREE + 2,        // [2]: the softmax warps' reference votes of a tile (parity)
                         // FP8 only: a V slot's e4m3 pages have landed (before their widening), scale ring
                         VLAND = VOTE + 2, SCALE = VLAND + NSV,
                         END = FP8 ? SCALE + 16 : VOTE + 2;
};

// A finished piece, as its epilogue needs it.
struct PieceDesc {
    int b, hg, qoff, Q, S0, S1, pc, pb;
    bool last;
};

struct Ctl {
    volatile int* abort;
    int* err;
    uint64_t limit_ns;     // the launch's wait limit (AttnParams::wait_limit_ns)
};

// Bounded wait: spins on try_wait; gives up after the launch's wait limit or
// once the CTA's abort flag is set.  A timeout raises PKV_DEVERR_TIMEOUT and
// the flag.  The spin loop is out of line: only the first try sits in the
// callers' code.
__device__ __noinline__ bool wait_bar_spin(uint32_t bar, uint32_t parity, volatile int* abort, int* err,
                                           uint64_t limit_ns) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63) == 0) {
            if (*abort) return false;
            if (globaltimer_ns() - t0 > limit_ns) {
                raise_error(err, PKV_DEVERR_TIMEOUT);
                *abort = 1;
                return false;
            }
        }
    }
}
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const Ctl& c) {
    if (mbar_try_wait(bar, parity)) return true;
    return wait_bar_spin(bar, parity, c.abort, c.err, c.limit_ns);
}

// 2^x by the SFU (flushes subnormal results to zero, 2^-inf = 0).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}

// OR of v over the n threads of named barrier `id` (one role, uniform
// control flow: the .aligned form, like named_bar_sync).
__device__ __forceinline__ bool bar_red_or(int id, int n, bool v) {
    uint32_t r;
    asm volatile(
        "{\n.reg .pred p, q;\nsetp.ne.u32 q, %1, 0;\nbar.red.or.pred p, %2, %3, q;\nselp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}

// Reduction (sum or max) of N per-lane columns over aligned groups of lanes,
// by exchanges with lane ^ S for S = G/2 .. 1 (G the group size): at each
// exchange a lane keeps half of its columns and receives the partner's values
// of that half, so the whole reduction takes N - 1 shuffles (plus one per
// exchange once a single column is left) instead of N log2(G).  On return
// a[0] holds the group's result for column col (N <= G; lanes that differ only
// in the bits below log2(G / N) hold the same column).
template <int N, int S, bool MAX>
struct Butterfly {
    static __device__ __forceinline__ void run(float* a, int lane, int& col) {
        if constexpr (N > 1) {
            constexpr int H = N / 2;
            const bool up = (lane & S) != 0;
#pragma unroll
            for (int j = 0; j < H; ++j) {
                const float send = up ? a[j] : a[H + j];
                const float keep = up ? a[H + j] : a[j];
                const float got = __shfl_xor_sync(0xffffffffu, send, S);
                a[j] = MAX ? fmaxf(keep, got) : keep + got;
            }
            if (up) col += H;
            if constexpr (S > 1) Butterfly<H, S / 2, MAX>::run(a, lane, col);
        } else {
            const float got = __shfl_xor_sync(0xffffffffu, a[0], S);
            a[0] = MAX ? fmaxf(a[0], got) : a[0] + got;
            if constexpr (S > 1) Butterfly<1, S / 2, MAX>::run(a, lane, col);
        }
    }
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// Four e4m3 codes (bytes of w, lowest first) -> four fp16 (lo: codes 0, 1;
// hi: codes 2, 3) by CUDA's conversion: exact (every e4m3 value is an fp16
// value), NaN codes to NaN.
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
    const __half2_raw a = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w & 0xffffu), __NV_E4M3);
    const __half2_raw b = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w >> 16), __NV_E4M3);
    lo = (uint32_t)a.x | ((uint32_t)a.y << 16);
    hi = (uint32_t)b.x | ((uint32_t)b.y << 16);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    const __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

// Pieces of a CTA's unit range [u0, u1), in processing order: the piece
// holding u1 - 1 first (when it does not start at u0), then [u0, start of
// that piece) front to back.  Segment = (sequence, group of HG kv-heads), its
// units = pages x HG in page-major order.  Every role walks it the same way.
template <bool CASC>
struct PieceIter {
    const int4* tab;            // per-sequence table in shared memory, or nullptr
    Cursor cur, fcur;
    int u, stop, u0, HG, Hkv;
    bool tail_phase;
    int hg, S0, S1, pg0, npg;   // current piece: group, segment [S0, S1), units [S0+pg0, S0+pg0+npg)

    __device__ void load_at(int uu, int end) {
        const int len = cur.nb * HG;
        hg = div_small(uu - cur.Ub, len);
        S0 = cur.Ub + hg * len;
        S1 = S0 + len;
        pg0 = uu - S0;
        npg = min(end, S1) - uu;
    }
    __device__ void init(const AttnParams& p, const Cursor& c0, const Cursor& ct, int u0_, int u1) {
        HG = p.hg;
        Hkv = p.num_kv_heads;
        u0 = u0_;
        fcur = c0;
        cur = ct;
        const int len = ct.nb * HG;
        const int s0t = ct.Ub + div_small(u1 - 1 - ct.Ub, len) * len;
        const int tstart = max(u0, s0t);
        if (tstart > u0) {
            tail_phase = true;
            stop = tstart;          // the forward walk ends where the tail piece starts
            u = tstart;
            load_at(tstart, u1);
        } else {
            tail_phase = false;
            stop = u1;
            cur = c0;
            u = u0;
            load_at(u0, u1);
        }
    }
    __device__ bool valid() const { return tail_phase || u < stop; }
    __device__ void advance(const AttnParams& p) {
        if (tail_phase) {
            tail_phase = false;
            cur = fcur;
            u = u0;
            load_at(u, stop);
            return;
        }
        u += npg;
        if (u < stop && u == cur.Ub + cur.nb * Hkv) cursor_next<CASC>(p, cur, tab);
        if (u < stop) load_at(u, stop);
    }
};

// Column n of segment (b, hg) -> element offset of its q / out row.
__device__ __forceinline__ size_t col_row_offset(const AttnParams& p, int qoff, int R, int hg, int n, int D) {
    const int hh = div_small(n, R), r = n - hh * R, i = div_small(r, p.group), hl = r - i * p.group;
    return ((size_t)(qoff + i) * p.num_q_heads + (hg * p.hg + hh) * p.group + hl) * D;
}

// One step of the online merge of split partials (m, l, a): the running
// (M, den, num) and the new piece are both brought to the larger reference.
// Written with explicit roundings so the merge gives the same bits wherever
// it is inlined.
__device__ __forceinline__ void merge_weights(float& M, float m, float& wo, float& wn) {
    const float mn = fmaxf(M, m);
    wo = (M == -INFINITY) ? 0.f : fast_exp2(M - mn);
    wn = (m == -INFINITY) ? 0.f : fast_exp2(m - mn);
    M = mn;
}
__device__ __forceinline__ float merge_acc(float x, float wo, float y, float wn) {
    return __fmaf_rn(y, wn, __fmul_rn(x, wo));
}

// Final store of one output element: the row at element offset `off` of
// out (sequence row, query head, dim 0), dim d, value num / den with
// reference max M (log2 units).  In a cascade's prefix pass the value and
// its log2-sum-exp M + log2(den) go to the state arrays instead; in its
// suffix pass a row whose sequence has a group prefix (pb > 0) is merged
// with that prefix state first (the same LSE rule as the split merge).
template <int D, bool CASC>
__device__ __forceinline__ void store_out(const AttnParams& p, size_t off, int d, float num, float den, float M,
                                          int pb) {
    const float o = __fdividef(num, den);
    if constexpr (!CASC) {                     // (the plain kernels carry none of the cascade's code)
        p.out[off + d] = __float2bfloat16_rn(o);
        return;
    }
    if (p.cascade == 1) {
        p.state_o[off + d] = o;
        if (d == 0) p.state_lse[off / D] = M + __log2f(den);
        return;
    }
    if (p.cascade == 2 && pb > 0) {
        const float ls = M + __log2f(den), lp = __ldcg(p.state_lse + off / D), op = __ldcg(p.state_o + off + d);
        const float mx = fmaxf(ls, lp), ws = fast_exp2(ls - mx), wp = fast_exp2(lp - mx);
        p.out[off + d] = __float2bfloat16_rn(__fdividef(__fmaf_rn(o, ws, __fmul_rn(op, wp)), ws + wp));
        return;
    }
    p.out[off + d] = __float2bfloat16_rn(o);
}

// Merge the partials of segment [S0, S1) (NCOL columns) into out; one warp,
// one round trip of loads per piece, pieces in CTA order.
template <int D, bool CASC>
__device__ void merge_segment_warp(const AttnParams& p, int hg, int qoff, int Q, int S0, int S1, const Part& part,
                                   int lane, int pb) {
    constexpr int DPL = D / 32;
    const int c_first = part.owner(S0), c_last = part.owner(S1 - 1);
    const int R = p.group * Q, ncol = p.hg * R;
    for (int n0 = 0; n0 < ncol; n0 += 8) {
        float M[8], den[8], num[8][DPL];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            M[k] = -INFINITY;
            den[k] = 0.f;
#pragma unroll
            for (int x = 0; x < DPL; ++x) num[k][x] = 0.f;
        }
        for (int c = c_first; c <= c_last; ++c) {
            const float* s = slot_ptr(p, c, S0, part.start(c));
            float m[8], l[8], a[8][DPL];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int n = n0 + k;
                m[k] = n < ncol ? __ldcg(s + n) : -INFINITY;
                l[k] = n < ncol ? __ldcg(s + p.rows_pad + n) : 0.f;
#pragma unroll
                for (int x = 0; x < DPL; ++x)
                    a[k][x] = n < ncol ? __ldcg(s + 2 * p.rows_pad + (size_t)n * D + lane + 32 * x) : 0.f;
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                float wo, wn;
                merge_weights(M[k], m[k], wo, wn);
                den[k] = merge_acc(den[k], wo, l[k], wn);
#pragma unroll
                for (int x = 0; x < DPL; ++x) num[k][x] = merge_acc(num[k][x], wo, a[k][x], wn);
            }
        }
        const size_t my_off = n0 + lane < ncol ? col_row_offset(p, qoff, R, hg, n0 + lane, D) : 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int n = n0 + k;
            const size_t off = __shfl_sync(0xffffffffu, my_off, k);
            if (n < ncol) {
#pragma unroll
                for (int x = 0; x < DPL; ++x) store_out<D, CASC>(p, off, lane + 32 * x, num[k][x], den[k], M[k], pb);
            }
        }
    }
}

// CASC: the instantiations a shared-prefix cascade launches (prefix pass:
// group rows, no causal mask, states out; suffix pass: a first page per
// sequence, rows merged with the prefix states); plain calls use CASC = false.
template <int D, int NPAD, bool SPLIT, int NSK, int NSV, bool EWG, bool FP8, bool CASC>
__global__ void __launch_bounds__(threads_of<EWG>(), 1) attn_tc_kernel(const AttnParams p) {
    using K = Cfg<D, NPAD, SPLIT, NSK, NSV, EWG, FP8>;
    using B = Bars<NSK, NSV, FP8>;
    static_assert(B::END == K::NBAR, "barrier count");
    static_assert(!FP8 || EWG, "FP8 V pages are widened by the epilogue warpgroup");
    constexpr int RMAX = K::RMAX;
    constexpr int kThreads = threads_of<EWG>();
    extern __shared__ uint8_t smem_raw[];
    __shared__ int scratch[kThreads / 32 + 1];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    const uint32_t sb = smem_u32(smem);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cta = blockIdx.x;
    // The kernel that follows on the stream may launch now: its CTAs take the
    // SMs this grid frees as its CTAs finish, and run their own set-up while
    // the last ones still stream (its dependency wait still holds back what
    // it reads from this grid's results).
    griddep_launch();
    // This CTA's sequence lengths, loaded first: their latency overlaps the
    // barrier, TMEM and Q-buffer set-up below.
    int2 lq = make_int2(0, 0);
    if (p.num_seqs <= kThreads && tid < p.num_seqs) lq = make_int2(__ldg(p.context_lens + tid), __ldg(p.q_lens + tid));

    auto bar = [&](int i) -> uint32_t { return sb + K::OFF_BAR + 8 * i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + K::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + K::OFF_MISC + 4);
    volatile int* never = reinterpret_cast<volatile int*>(smem + K::OFF_MISC + 8);   // stays 0
    // pre-merge of the last piece's segment: 0 open, 1 the merge warp gathers, 2 gathered,
    // 3 the epilogue went its own way
    volatile int* gstate = reinterpret_cast<volatile int*>(smem + K::OFF_MISC + 12);
    float* gbuf = reinterpret_cast<float*>(smem + K::OFF_GATHER);
    float* lred = reinterpret_cast<float*>(smem + K::OFF_LRED);   // [2][4][RMAX]
    float* emref = reinterpret_cast<float*>(smem + K::OFF_EM);    // [2][RMAX]
    int* pdesc = reinterpret_cast<int*>(smem + K::OFF_PD);        // [2][8]
    const Ctl ctl{abort_flag, p.err, p.wait_limit_ns};
    const Ctl drain{never, p.err, p.wait_limit_ns};      // bounded waits that ignore the abort flag

    // Q buffers start zeroed: rows past a piece's columns are never written
    // and only feed S^T columns the softmax ignores.
    for (int i = tid; i < 2 * K::QBUF / 16; i += kThreads)
        reinterpret_cast<uint4*>(smem + K::OFF_Q)[i] = make_uint4(0, 0, 0, 0);
    if constexpr (FP8)   // (scale slots of units past a tile's pages are read, never used)
        for (int i = tid; i < K::NSC * 128 / 16; i += kThreads)
            reinterpret_cast<uint4*>(smem + K::OFF_SC)[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    if (tid == 0) {
        // K slots are filled by bulk copies (bf16 or e4m3 pages); V slots too, or
        // (FP8) by the epilogue warpgroup's widening (all 128 threads arrive)
        for (int s = 0; s < NSK; ++s) {
            mbar_init(bar(B::KFULL + s), 1);
            mbar_init(bar(B::KEMPTY + s), 1);
        }
        for (int s = 0; s < NSV; ++s) {
            mbar_init(bar(B::VFULL + s), FP8 ? kSoftThreads : 1);
            mbar_init(bar(B::VEMPTY + s), 1);
        }
        if constexpr (FP8) {
            for (int s = 0; s < NSV; ++s) mbar_init(bar(B::VLAND + s), 1);
            for (int s = 0; s < K::NSC; ++s) mbar_init(bar(B::SCALE + s), 33);   // 32 cp.async lanes + 1
        }
        for (int i = 0; i < NSB; ++i) {
            mbar_init(bar(B::SFULL + i), 1);
            mbar_init(bar(B::PFULL + i), kSoftThreads);
            mbar_init(bar(B::PEMPTY + i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(B::QFULL + i), 1);
            mbar_init(bar(B::QEMPTY + i), 1);
            mbar_init(bar(B::ODONE + i), 1);
            mbar_init(bar(B::PREADY + i), kSoftThreads);
            mbar_init(bar(B::OFREE + i), kSoftThreads);
            mbar_init(bar(B::VOTE + i), 4);                 // lane 0 of each softmax warp
        }
        mbar_init(bar(B::DONE), 1);
        mbar_init(bar(B::DONE + 1), 1);
        for (int i = 0; i < 4; ++i) mbar_init(bar(B::MQFULL + i), kSoftThreads);
        *abort_flag = 0;
        *never = 0;
        *gstate = 0;
        mbar_fence_init();
    }
    // The tensor memory is taken before the dependency wait too.
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), K::TMEM_COLS);
        tmem_relinquish();
    }
    // Under a programmatic dependent launch this kernel starts while the
    // previous kernel on the stream (the step's append) still runs.  The
    // planning reads only caller inputs that kernel does not write (lengths,
    // block tables, q), so it runs at once; the producer waits for the
    // previous kernel's writes to be visible before its first K/V copy, and
    // the merge warp before it touches the workspace.
    Cursor cur0, curt;
    int u0, u1, W, P;
    int4* seqtab = p.num_seqs <= K::SEQTAB ? reinterpret_cast<int4*>(smem + K::OFF_SEQ) : nullptr;
    // Wide and FP8 segments cut the CTA ranges by weight: every segment is
    // charged a fixed number of units on top of its own for what a piece costs
    // beyond its bytes (its partial last tile, which takes a whole tile's time,
    // the piece start and, for wide segments, the epilogue in the softmax warps:
    // about three tiles).  Narrow bf16 segments keep the equal split, which
    // needs no table at the start (the table cost them ~2 us a launch).
    int* bndtab = K::PTAB ? reinterpret_cast<int*>(smem + K::OFF_BND) : nullptr;
    bool tab_used = false;
    const bool has_work = plan_locate<kThreads, CASC>(p, blockIdx.x, gridDim.x, scratch, &cur0, &u0, &u1, &W, &P, &curt,
                                                seqtab, bndtab, K::TABMAX, SPLIT ? kNarrowCharge : EWG ? kWideEwgCharge : 24, &tab_used,
                                                reinterpret_cast<int4*>(smem + K::OFF_P),   // (P ring unused yet)
                                                CASC ? nullptr : &lq);
    const Part part{W, P, tab_used ? bndtab : nullptr};
    if (!has_work) {             // uniform across the CTA
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (warp == 0) tmem_dealloc(*tmem_slot, K::TMEM_COLS);
        return;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int G = p.group, Hkv = p.num_kv_heads, HG = p.hg;

    PieceIter<CASC> it;
    it.tab = seqtab;
    it.init(p, cur0, curt, u0, u1);

    // ---------------------------------------------------------------- FP8 widening
    // Tiles of the CTA (every role walks the same pieces).
    auto tile_count = [&]() {
        int n = 0;
        PieceIter<CASC> w = it;
        while (w.valid()) {
            n += (w.npg + kTP - 1) / kTP;
            w.advance(p);
        }
        return n;
    };
    // Widen one operand slot in place: the bulk copy left the tile's e4m3 pages
    // (layout [2][D/16][8][16] bytes) in the slot's upper half.  Each thread of
    // a 128-thread warpgroup (named barrier bid) reads its 16-byte chunk e of
    // NPT of the pages (D = 128: chunk tt of all 8 pages; D = 64, 64 chunks a
    // page: chunk tt % 64 of pages tt / 64, tt / 64 + 2, ...), the warpgroup
    // syncs, then writes the fp16 operand ([2][D/8][8][8] elements per page)
    // over the whole slot.  Codes are exact in fp16 (NaN codes become NaN);
    // the page scales are applied in the softmax (P carries the v scale).
    auto widen = [&](uint8_t* slot, int tt, int bid) {
        constexpr int CPP8 = K::PAGE8 / 16;                  // 16-byte chunks of an e4m3 page
        constexpr int PSTEP = kSoftThreads / CPP8;           // pages between a thread's pages
        constexpr int NPT = kTP / PSTEP;                     // pages a thread widens
        static_assert(!FP8 || (kSoftThreads % CPP8 == 0 && kTP % PSTEP == 0), "widening split");
        constexpr int NC16 = D / 16;
        const int e = tt % CPP8, k0 = tt / CPP8;
        uint4 v[NPT];
#pragma unroll
        for (int j = 0; j < NPT; ++j)
            v[j] = *reinterpret_cast<const uint4*>(slot + K::OFF_LAND + (k0 + j * PSTEP) * K::PAGE8 + e * 16);
        named_bar_sync(bid, kSoftThreads);
        // chunk e of a page: token group e / (8 NC16), 16-element column block (e / 8) % NC16, token e % 8
        const int r = e & 7, c = (e >> 3) % NC16, oh = e / (8 * NC16);
        uint8_t* d0 = slot + ((oh * (D / 8) + 2 * c) * 8 + r) * 16 + k0 * K::PAGE;
#pragma unroll
        for (int j = 0; j < NPT; ++j) {
            const uint32_t wv[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
            uint32_t o[8];
#pragma unroll
            for (int x = 0; x < 4; ++x) e4m3x4_to_f16x4(wv[x], o[2 * x], o[2 * x + 1]);
            *reinterpret_cast<uint4*>(d0 + j * PSTEP * K::PAGE) = make_uint4(o[0], o[1], o[2], o[3]);
            *reinterpret_cast<uint4*>(d0 + j * PSTEP * K::PAGE + 128) = make_uint4(o[4], o[5], o[6], o[7]);
        }
        fence_proxy_async_smem();             // the MMA reads the slot through the async proxy
    };

    // ---------------------------------------------------------------- piece epilogue
    // Run by one warpgroup (thread tt = TMEM lane = d row, named barrier bid)
    // once piece d's column sums and reference max are in lred / emref (parity
    // d.pc & 1): waits for the piece's last P.V, reads O^T, then writes the
    // output (complete segment), or hands the partial to the merge warp (a
    // split piece before the CTA's last), or closes the segment (the last
    // piece: the merge warp's pre-merge, a direct merge when every other piece
    // is published, else publish and draw the ticket).  With EWG the O^T and
    // smem reads end with an arrive on OFREE, which frees them for piece d.pc + 2.
    int n_tasks = 0;
    auto piece_epilogue = [&](const PieceDesc& d, int tt, int bid) {
        const int lanee = tt & 31;
        const uint32_t lbase = (uint32_t)((tt >> 5) * 32) << 16;
        const bool complete = (d.S0 >= u0) && (d.S1 <= u1);
        const int R = G * d.Q, ncol = HG * R, par = d.pc & 1;
        int* ticket = p.tickets + d.b * Hkv + d.hg;
        // the CTA's last piece, ending its segment: take the merge warp's pre-merge
        // when it is there (or about to be), else close the pre-merge to it
        const bool gather_ok = SPLIT && !complete && d.last && d.S0 < u0 && d.S1 <= u1;
        int tk = -1, gs = 0;
        if (!complete && d.last && tt == 0) {
            if (gather_ok) {
                gs = atomicCAS(const_cast<int*>(gstate), 0, 3);
                if (gs == 1) {
                    const uint64_t g0 = globaltimer_ns();
                    while ((gs = *gstate) == 1 && !*abort_flag) {
                        if (globaltimer_ns() - g0 > p.wait_limit_ns) {
                            raise_error(p.err, PKV_DEVERR_TIMEOUT);
                            *abort_flag = 1;
                        }
                    }
                }
                __threadfence_block();
            }
            // the segment's ticket, read without blocking: its latency overlaps the wait
            // for the piece's last P.V and the O^T read (an acquire fence follows only
            // if it shows every other piece published)
            if (gs != 2) tk = ld_relaxed_gpu(ticket);
        }
        named_bar_sync(bid, kSoftThreads);          // (the piece-end sums of all four warps)
        wait_bar(bar(B::ODONE + par), (d.pc >> 1) & 1, ctl);
        tc_fence_after();
        float acc[RMAX], Lsum[RMAX], Mx[RMAX];
        {
            // column n belongs to kv-head n / R of the segment and sits in that head's accumulator
#pragma unroll
            for (int n = 0; n < RMAX; ++n) acc[n] = 0.f;
            for (int hh = 0; hh < HG; ++hh) {
                float o[K::NM];
#pragma unroll
                for (int c = 0; c < K::NM; c += 16) {
                    float tmp[16];
                    tmem_ld16(tmem + lbase + K::COL_O + (par * K::HGMAX + hh) * K::NM + c, tmp);
#pragma unroll
                    for (int x = 0; x < 16; ++x) o[c + x] = tmp[x];
                }
#pragma unroll
                for (int n = 0; n < RMAX; ++n)
                    if (n >= hh * R && n < hh * R + R) acc[n] = SPLIT ? (o[2 * n] + o[2 * n + 1]) : o[n];
            }
            const float* lw = lred + par * 4 * RMAX;
#pragma unroll
            for (int n = 0; n < RMAX; ++n) {
                Mx[n] = emref[par * RMAX + n];
                Lsum[n] = lw[n] + lw[RMAX + n] + lw[2 * RMAX + n] + lw[3 * RMAX + n];
                // no visible token of the piece reached column n: its head's accumulator may
                // not even have been started in this piece
                if (Mx[n] == -INFINITY) acc[n] = 0.f;
            }
        }
        tc_fence_before();
        if constexpr (EWG) mbar_arrive(bar(B::OFREE + par));   // O^T, lred and emref of this parity are read
        // column n's output row offset, computed by lane n and broadcast
        const size_t my_off = lanee < ncol ? col_row_offset(p, d.qoff, R, d.hg, lanee, D) : 0;
        if (complete) {
#pragma unroll
            for (int n = 0; n < RMAX; ++n) {
                const size_t off = __shfl_sync(0xffffffffu, my_off, n);
                if (n < ncol && tt < D) store_out<D, CASC>(p, off, tt, acc[n], Lsum[n], Mx[n], d.pb);
            }
            return;
        }
        if constexpr (SPLIT) {
            if (bar_red_or(bid, kSoftThreads, gs == 2)) {
                // the earlier pieces arrive pre-merged; add this one, the last in CTA order
#pragma unroll
                for (int n = 0; n < RMAX; ++n) {
                    float M = gbuf[n], den = gbuf[RMAX + n];
                    float num = tt < D ? gbuf[2 * RMAX + n * D + tt] : 0.f;
                    float wo, wn;
                    merge_weights(M, Mx[n], wo, wn);
                    den = merge_acc(den, wo, Lsum[n], wn);
                    num = merge_acc(num, wo, acc[n], wn);
                    const size_t off = __shfl_sync(0xffffffffu, my_off, n);
                    if (n < ncol && tt < D) store_out<D, CASC>(p, off, tt, num, den, M, d.pb);
                }
                return;
            }
        }
        const int c_first = d.last ? part.owner(d.S0) : 0;
        const int c_last = d.last ? part.owner(d.S1 - 1) : 0;
        // the last piece merges here when every other piece is published already
        if (tt == 0 && tk == c_last - c_first) fence_acquire_gpu();
        bool direct = d.last && bar_red_or(bid, kSoftThreads, tk == c_last - c_first);
        if (!direct) {
            float* slot = slot_ptr(p, cta, d.S0, u0);
#pragma unroll
            for (int n = 0; n < RMAX; ++n) {
                if (n < ncol) {
                    if (tt == n) {
                        slot[n] = Mx[n];
                        slot[p.rows_pad + n] = Lsum[n];
                    }
                    if (tt < D) slot[2 * p.rows_pad + (size_t)n * D + tt] = acc[n];
                }
            }
            if (!d.last) {
                // hand it to the merge warp (a CTA range cuts at most two segments, so the
                // 4-entry task ring never wraps onto a pending task)
                if (tt == 0) {
                    int* task = reinterpret_cast<int*>(smem + K::OFF_MQ) + (n_tasks & 3) * 8;
                    task[0] = d.b;
                    task[1] = d.hg;
                    task[2] = d.qoff;
                    task[3] = d.Q;
                    task[4] = d.S0;
                    task[5] = d.S1;
                    task[6] = d.pb;
                }
                mbar_arrive(bar(B::MQFULL + (n_tasks & 3)));
                ++n_tasks;
                return;
            }
            // the last piece: publish here and draw the ticket
            named_bar_sync(bid, kSoftThreads);     // every thread's part is stored
            int lst = 0;
            if (tt == 0) lst = atom_add_acq_rel_gpu(ticket, 1) == c_last - c_first;
            direct = bar_red_or(bid, kSoftThreads, lst != 0);
        }
        if (direct) {
            // merge in CTA order, this piece from registers (the same steps as
            // merge_segment_warp, so either place gives the same bits)
#pragma unroll
            for (int n0 = 0; n0 < RMAX; n0 += 8) {
                if (n0 >= ncol) break;
                float M[8], den[8], num[8];
#pragma unroll
                for (int x = 0; x < 8; ++x) {
                    M[x] = -INFINITY;
                    den[x] = 0.f;
                    num[x] = 0.f;
                }
                // the partials of MB CTAs at a time: every load in flight before the first is
                // used (at the launch's end these reads queue behind the other CTAs' streams)
                constexpr int MB = FP8 ? 2 : 1;
                for (int cb = c_first; cb <= c_last; cb += MB) {
                    float m[MB][8], l[MB][8], a[MB][8];
#pragma unroll
                    for (int j = 0; j < MB; ++j) {
                        const int c = cb + j;
                        if (c == cta) {
#pragma unroll
                            for (int x = 0; x < 8; ++x) {      // (RMAX may end inside a group of 8)
                                m[j][x] = n0 + x < RMAX ? Mx[n0 + x] : -INFINITY;
                                l[j][x] = n0 + x < RMAX ? Lsum[n0 + x] : 0.f;
                                a[j][x] = n0 + x < RMAX ? acc[n0 + x] : 0.f;
                            }
                        } else {
                            const bool cok = c <= c_last;
                            const float* sl = slot_ptr(p, cok ? c : cta, d.S0, part.start(cok ? c : cta));
#pragma unroll
                            for (int x = 0; x < 8; ++x) {
                                const int n = n0 + x;
                                m[j][x] = cok && n < ncol ? __ldcg(sl + n) : -INFINITY;
                                l[j][x] = cok && n < ncol ? __ldcg(sl + p.rows_pad + n) : 0.f;
                                a[j][x] = (cok && n < ncol && tt < D) ? __ldcg(sl + 2 * p.rows_pad + (size_t)n * D + tt) : 0.f;
                            }
                        }
                    }
#pragma unroll
                    for (int j = 0; j < MB; ++j) {
                        if (cb + j > c_last) break;
#pragma unroll
                        for (int x = 0; x < 8; ++x) {
                            float wo, wn;
                            merge_weights(M[x], m[j][x], wo, wn);
                            den[x] = merge_acc(den[x], wo, l[j][x], wn);
                            num[x] = merge_acc(num[x], wo, a[j][x], wn);
                        }
                    }
                }
#pragma unroll
                for (int x = 0; x < 8; ++x) {
                    const int n = n0 + x;
                    const size_t off = __shfl_sync(0xffffffffu, my_off, n);
                    if (n < ncol && tt < D) store_out<D, CASC>(p, off, tt, num[x], den[x], M[x], d.pb);
                }
            }
            if (tt == 0) *ticket = 0;              // ready for the next launch
        }
    };

    if (warp == kProducerWarp) {
        // ------------------------------------------------------------ producer
        // Runs one piece ahead on its inputs: once a piece's first tile is on
        // its way, the q rows and the first block-table window of the next piece
        // are loaded, and within a piece the next 32-page window of the block
        // table is loaded while the current one is used, so no copy waits on a
        // table read after the first.
        const uint64_t pol = policy_evict_first();
        constexpr int QV = (RMAX * K::NCH + 31) / 32;
        constexpr bool kQAhead = QV <= 4;         // wide pieces load their q at the piece start
        int t = 0, j = 0, kcount = 0, vcount = 0;
        bool ok = true;
        float cur_c = 1.f;                // (FP8) lane n < RMAX: column n's factor 2^-E_n in the current piece
        // q rows of piece `pi` in column order, 16 bytes per lane and step
        auto load_q = [&](const PieceIter<CASC>& pi, uint4 (&v)[QV]) {
            const int R = G * pi.cur.Q, ncol = HG * R;
#pragma unroll
            for (int k = 0; k < QV; ++k) {
                const int idx = lane + 32 * k;
                v[k] = make_uint4(0, 0, 0, 0);
                if (idx < ncol * K::NCH) {
                    const int n = idx / K::NCH, c = idx % K::NCH;
                    v[k] = __ldg(reinterpret_cast<const uint4*>(p.q + col_row_offset(p, pi.cur.qoff, R, pi.hg, n, D) +
                                                                c * 8));
                }
            }
        };
        // block-table entries [ws, ws + 32) of piece `pi`'s sequence, entry ws + lane per lane
        auto load_win = [&](const PieceIter<CASC>& pi, int ws) -> int {
            // (a cascade's prefix pass reads its group's first sequence's row; a suffix
            // pass starts after the group prefix's pages)
            const int row = (CASC && p.cascade == 1) ? __ldg(p.group_starts + pi.cur.b) : pi.cur.b;
            const int32_t* table = p.block_tables + (size_t)row * p.max_blocks_per_seq + (CASC ? pi.cur.pb : 0);
            return ws + lane < pi.cur.nb ? __ldg(table + ws + lane) : 0;
        };
        uint4 qv[QV];
        int win = 0;
        if (it.valid()) {
            if constexpr (kQAhead) load_q(it, qv);
            win = load_win(it, div_small(it.pg0, HG));
        }
        griddep_wait();                   // K/V pages the previous kernel wrote are visible from here
        if (p.hold != nullptr && it.valid()) {
            // (tests of the timeout path only) wait, bounded, for a flag; nothing sets the
            // flag the tests pass, so the wait runs out and every role winds down
            bool w = true;
            if (lane == 0) {
                const uint64_t h0 = globaltimer_ns();
                while (*reinterpret_cast<const volatile int*>(p.hold) == 0) {
                    if (*abort_flag) {
                        w = false;
                        break;
                    }
                    if (globaltimer_ns() - h0 > p.wait_limit_ns) {
                        raise_error(p.err, PKV_DEVERR_TIMEOUT);
                        *abort_flag = 1;
                        w = false;
                        break;
                    }
                    __nanosleep(256);
                }
            }
            ok = __shfl_sync(0xffffffffu, w, 0);
        }
        while (ok && it.valid()) {
            PieceIter<CASC> nx = it;
            uint4 qn[kQAhead ? QV : 1];
            int winn = 0;
            if constexpr (!kQAhead) load_q(it, qv);
            const int qb = j & 1;
            if (j >= 2) {
                bool w = lane == 0 ? wait_bar(bar(B::QEMPTY + qb), ((j >> 1) - 1) & 1, ctl) : true;
                ok = __shfl_sync(0xffffffffu, w, 0);
                if (!ok) break;
            }
            const int R = G * it.cur.Q, ncol = HG * R;
            int ws = div_small(it.pg0, HG);                        // win: entries [ws, ws + 32); win2: the next 32
            int win2 = 0;                                 // (loaded after the first tile, which stays in win)
            for (int t0 = 0; t0 < it.npg; t0 += kTP, ++t) {
                const int np = min(kTP, it.npg - t0);
                const int ks = t % NSK, vs = t % NSV;
                const int qfirst = it.pg0 + t0;                       // first unit of the tile
                const int qu = qfirst + (lane & 7);
                const int qpg = div_small(qu, HG);                    // page of the lane's unit
                const int pg = qpg - ws;                          // in [0, 40) for the tile's units
                int blk = __shfl_sync(0xffffffffu, win, pg & 31);
                // the next window's entries only once the tile reaches them (its load may be in flight)
                if (div_small(qfirst + np - 1, HG) - ws >= 32) {
                    const int e2 = __shfl_sync(0xffffffffu, win2, pg & 31);
                    if (pg >= 32) blk = e2;
                }
                if (blk < 0 || blk >= p.num_blocks) {
                    if (lane < np) raise_error(p.err, PKV_DEVERR_BLOCK_ID);      // (lane < 8 here)
                    blk = 0;
                }
                const int qh = qu - qpg * HG;                         // the unit's head within the group
                const size_t unit = (size_t)blk * p.cache_kv_heads + cache_head(p, it.hg * HG + qh);
                const size_t off = unit * (FP8 ? K::PAGE8 : K::PAGE);
                // K and V of the tile in one pass: lanes 0-7 copy K, lanes 8-15 V (unit slot
                // lane & 7).  One bulk copy per page: the group's heads of a block are adjacent
                // in the cache and the tile, so the lane of a page's first unit copies its run.
                const int sl = lane & 7, kv = lane >> 3;
                const bool lead = kv < 2 && sl < np && (sl == 0 || qh == 0);
                const int run = min(HG - qh, np - sl);
                {
                    bool w = true;
                    if (lane == 0 && t >= NSK) w = wait_bar(bar(B::KEMPTY + ks), ((t / NSK) - 1) & 1, ctl);
                    if (lane == 8 && t >= NSV) w = wait_bar(bar(B::VEMPTY + vs), ((t / NSV) - 1) & 1, ctl);
                    ok = __all_sync(0xffffffffu, w);
                    if (!ok) break;
                }
                {
                    // (FP8: the S MMA reads the e4m3 K pages; V lands in its slot's upper half)
                    constexpr int KP = FP8 ? K::PAGE8 : K::PAGE;
                    const uint32_t vslot = sb + K::OFF_V + vs * (K::TILE + K::VSLACK) + (FP8 ? K::OFF_LAND : 0);
                    const uint32_t fb = kv == 0 ? bar(B::KFULL + ks) : bar((FP8 ? B::VLAND : B::VFULL) + vs);
                    if (sl == 0 && kv < 2) mbar_arrive_expect_tx(fb, np * KP);
                    __syncwarp();
                    if (lead)
                        bulk_g2s_hint(kv == 0 ? sb + K::OFF_K + ks * K::KSLOT + sl * KP : vslot + sl * KP,
                                      (kv == 0 ? p.k_cache : p.v_cache) + off, run * KP, fb, pol);
                }
                ++kcount;
                if (t0 == 0) {
                    // the piece's q rows -> Q buffer (K-major core matrices)
                    uint8_t* qdst = smem + K::OFF_Q + qb * K::QBUF;
                    if constexpr (FP8) {
                        // e4m3 operand of the S MMA: row n times 2^E_n (its largest magnitude
                        // brought to [128, 256)), split exactly into hi + lo e4m3 terms (a
                        // bf16 value's 8 significant bits), stored as rows n and 8 + n; the
                        // softmax adds the two columns and multiplies by 2^-E_n
                        static_assert(!FP8 || ((K::NCH == 16 || K::NCH == 8) && (RMAX == 8 || RMAX == 16)),
                                      "FP8 q staging: R <= 16");
                        int ek[QV];
#pragma unroll
                        for (int k = 0; k < QV; ++k) {
                            const uint32_t wq[4] = {qv[k].x, qv[k].y, qv[k].z, qv[k].w};
                            float mx = 0.f;
#pragma unroll
                            for (int h = 0; h < 4; ++h)
                                mx = fmaxf(mx, fmaxf(fabsf(__uint_as_float(wq[h] << 16)),
                                                     fabsf(__uint_as_float(wq[h] & 0xFFFF0000u))));
#pragma unroll
                            for (int o = K::NCH / 2; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                            const int e = (int)((__float_as_uint(mx) >> 23) & 0xFF) - 127;
                            const int E = mx > 0.f ? min(126, max(-126, 7 - e)) : 0;
                            ek[k] = E;
                            const float sf = __uint_as_float((uint32_t)(E + 127) << 23);
                            const int idx = lane + 32 * k;
                            if (idx < ncol * K::NCH) {
                                uint32_t hi[2] = {0u, 0u}, lo[2] = {0u, 0u};
#pragma unroll
                                for (int h = 0; h < 4; ++h) {
                                    const float x0 = __uint_as_float(wq[h] << 16) * sf;
                                    const float x1 = __uint_as_float(wq[h] & 0xFFFF0000u) * sf;
                                    const uint32_t c1 = __nv_cvt_float2_to_fp8x2(make_float2(x0, x1), __NV_SATFINITE, __NV_E4M3);
                                    const float2 b1 = e4m3x2_to_float2(c1);
                                    const uint32_t c2 =
                                        __nv_cvt_float2_to_fp8x2(make_float2(x0 - b1.x, x1 - b1.y), __NV_SATFINITE, __NV_E4M3);
                                    hi[h >> 1] |= (c1 & 0xFFFFu) << ((h & 1) * 16);
                                    lo[h >> 1] |= (c2 & 0xFFFFu) << ((h & 1) * 16);
                                }
                                const int n = idx / K::NCH, c = idx % K::NCH;    // row, 8-element chunk
                                // (8-row core-matrix groups (D / 16) * 128 bytes apart: rows n, then RMAX + n)
                                uint8_t* rh = qdst + (n >> 3) * ((D / 16) * 128) + (c >> 1) * 128 + (n & 7) * 16 + (c & 1) * 8;
                                *reinterpret_cast<uint2*>(rh) = make_uint2(hi[0], hi[1]);
                                *reinterpret_cast<uint2*>(rh + (RMAX / 8) * ((D / 16) * 128)) = make_uint2(lo[0], lo[1]);
                            }
                        }
                        // column n's factor -> lane n: a step holds RPS rows, row n in lanes
                        // (n % RPS) * NCH + [0, NCH) of step n / RPS
                        constexpr int RPS = 32 / K::NCH;
                        int en = 0;
#pragma unroll
                        for (int k = 0; k < QV; ++k) {
                            const int v = __shfl_sync(0xffffffffu, ek[k], (lane % RPS) * K::NCH);
                            if (lane / RPS == k) en = v;
                        }
                        cur_c = __uint_as_float((uint32_t)(127 - en) << 23);
                    } else {
#pragma unroll
                        for (int k = 0; k < QV; ++k) {
                            const int idx = lane + 32 * k;
                            if (idx < ncol * K::NCH) {
                                const int n = idx / K::NCH, c = idx % K::NCH;
                                *reinterpret_cast<uint4*>(qdst + (n >> 3) * (K::NCH * 128) + c * 128 + (n & 7) * 16) =
                                    qv[k];
                            }
                        }
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(B::QFULL + qb));
                }
                if constexpr (FP8) {
                    // this tile's (block, kv-head) scales straight into the scale ring (cp.async,
                    // each lane's arrival once its copies land) and the columns' factors (lane 0's
                    // arrival after the warp's stores): 33 arrivals complete the slot
                    const int ssl = t % K::NSC;
                    const uint32_t scs = sb + K::OFF_SC + ssl * 128;
                    if (lane < np) {
                        cp_async_4(scs + lane * 4, p.k_scales + unit);
                        cp_async_4(scs + 32 + lane * 4, p.v_scales + unit);
                    }
                    cp_async_mbar_arrive_noinc(bar(B::SCALE + ssl));
                    if (lane < RMAX) reinterpret_cast<float*>(smem + K::OFF_SC)[ssl * 32 + 16 + lane] = cur_c;
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(B::SCALE + ssl));
                }
                ++vcount;
                __syncwarp();
                if (t0 == 0) {
                    // look-ahead, once the piece's first tile is on its way
                    win2 = load_win(it, ws + 32);
                    nx.advance(p);
                    if (nx.valid()) {
                        if constexpr (kQAhead) load_q(nx, qn);
                        winn = load_win(nx, div_small(nx.pg0, HG));
                    }
                }
                // slide the table window once a tile has reached the next one
                if (div_small(qfirst + np - 1, HG) - ws >= 32 && t0 + kTP < it.npg) {
                    ws += 32;
                    win = win2;
                    win2 = load_win(it, ws + 32);
                }
            }
            ++j;
            it = nx;
            if constexpr (kQAhead) {
#pragma unroll
                for (int k = 0; k < QV; ++k) qv[k] = qn[k];
            }
            win = winn;
        }
        // drain: every copy issued has landed before the CTA exits
        if constexpr (FP8) cp_async_wait_all();
        if (lane == 0) {
            for (int tt = max(0, kcount - NSK); tt < kcount; ++tt)
                wait_bar(bar(B::KFULL + tt % NSK), (tt / NSK) & 1, drain);
            for (int tt = max(0, vcount - NSV); tt < vcount; ++tt)
                wait_bar(bar((FP8 ? B::VLAND : B::VFULL) + tt % NSV), (tt / NSV) & 1, drain);
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ S^T issuer
        // S^T of tile t once its K and its piece's q have landed and the
        // softmax has released S^T buffer t % NSB (P of tile t - NSB written).
        if (lane == 0) {
            constexpr uint32_t idS = FP8 ? idesc_e4m3_f32(128, K::NM) : idesc_bf16_f32(128, K::NM, false, false);
            constexpr int SBO = FP8 ? (D / 16) * 128 : K::NCH * 128;   // between 8-row core-matrix groups
            int t = 0, j = 0;
            bool ok = true;
            while (ok && it.valid()) {
                const int qb = j & 1;
                if (!(ok = wait_bar(bar(B::QFULL + qb), (j >> 1) & 1, ctl))) break;
                const uint32_t qbase = sb + K::OFF_Q + qb * K::QBUF;
                for (int t0 = 0; t0 < it.npg; t0 += kTP, ++t) {
                    const int ks = t % NSK;
                    if (t >= NSB && !(ok = wait_bar(bar(B::PFULL + t % NSB), ((t / NSB) - 1) & 1, ctl))) break;
                    if (!(ok = wait_bar(bar(B::KFULL + ks), (t / NSK) & 1, ctl))) break;
                    tc_fence_after();
                    const uint32_t kbase = sb + K::OFF_K + ks * K::KSLOT;
                    // K steps of 32 bytes (16 bf16 or 32 e4m3 elements), two core matrices each
#pragma unroll
                    for (int k = 0; k < (FP8 ? D / 32 : D / 16); ++k) {
                        const uint64_t a = smem_desc(kbase + k * 256, 128, SBO);
                        const uint64_t b = smem_desc(qbase + k * 256, 128, SBO);
                        if constexpr (FP8)
                            mma_f8(tmem + K::COL_S + (t % NSB) * K::NM, a, b, idS, k > 0);
                        else
                            mma_bf16(tmem + K::COL_S + (t % NSB) * K::NM, a, b, idS, k > 0);
                    }
                    mma_commit(bar(B::SFULL + t % NSB));
                    mma_commit(bar(B::KEMPTY + ks));
                    if (t0 + kTP >= it.npg) mma_commit(bar(B::QEMPTY + qb));
                }
                ++j;
                if (ok) it.advance(p);
            }
            mma_commit(bar(B::DONE));
            wait_bar(bar(B::DONE), 0, drain);
        }
        __syncwarp();
    } else if (warp == kPvWarp) {
        // ------------------------------------------------------------ P.V issuer
        // O^T += V^T P^T of tile t once its P is written and its V has landed;
        // pieces alternate between two accumulators, and a piece's first tile
        // starts its accumulator afresh once the epilogue of the piece two
        // before has read it.
        if (lane == 0) {
            // (FP8: fp16 operands, V widened to fp16)
            constexpr uint32_t idPV = FP8 ? idesc_f16_f32(128, K::NM, true, true) : idesc_bf16_f32(128, K::NM, true, true);
            int t = 0, pc = 0;
            bool ok = true;
            while (ok && it.valid()) {
                const uint32_t obase = tmem + K::COL_O + (pc & 1) * K::HGMAX * K::NM;
                uint32_t started = 0;             // kv-heads whose accumulator this piece has started
                if (EWG && pc >= 2 && !(ok = wait_bar(bar(B::OFREE + (pc & 1)), ((pc >> 1) - 1) & 1, ctl))) break;
                for (int t0 = 0; t0 < it.npg; t0 += kTP, ++t) {
                    const int np = min(kTP, it.npg - t0);
                    const int vs = t % NSV;
                    if (!(ok = wait_bar(bar(B::PFULL + t % NSB), (t / NSB) & 1, ctl))) break;
                    if (!(ok = wait_bar(bar(B::VFULL + vs), (t / NSV) & 1, ctl))) break;
                    tc_fence_after();
                    const uint32_t vbase = sb + K::OFF_V + vs * (K::TILE + K::VSLACK);
                    const uint32_t pbase = sb + K::OFF_P + (t % NSB) * K::PBUF;
                    // unit slot pg holds unit it.pg0 + t0 + pg of the segment: kv-head (hh0 + pg) % HG
                    const int hh0 = (it.pg0 + t0) - div_small(it.pg0 + t0, HG) * HG;
                    if constexpr (D == 64 && SPLIT && !FP8) {
                        // head_dim 64, bf16: slot order, so consecutive MMAs go to different heads'
                        // accumulators (one head's MMAs accumulate into the same columns one after
                        // another); this kernel's tiles are the shortest, and its P.V issuer had
                        // fallen ~2 tiles behind the softmax.  (The other kernels measured slower so.)
                        int hh = hh0;
                        for (int pg = 0; pg < np; ++pg) {
                            const uint32_t accum = (started >> hh) & 1u;
                            started |= 1u << hh;
                            mma_bf16(obase + hh * K::NM, smem_desc(vbase + pg * K::PAGE, K::NCH * 128, 128),
                                     smem_desc(pbase + pg * 256, 128, 16 * 128), idPV, accum);
                            if (++hh == HG) hh = 0;
                        }
                    } else {
                        for (int hh = 0; hh < HG; ++hh) {
                            const uint32_t ocol = obase + hh * K::NM;
                            for (int pg = hh >= hh0 ? hh - hh0 : hh - hh0 + HG; pg < np; pg += HG) {
                                const uint32_t accum = (started >> hh) & 1u;
                                started |= 1u << hh;
                                const uint64_t a = smem_desc(vbase + pg * K::PAGE, K::NCH * 128, 128);
                                const uint64_t b = smem_desc(pbase + pg * 256, 128, 16 * 128);
                                mma_bf16(ocol, a, b, idPV, accum);
                                if constexpr (!SPLIT) {      // (wide: P's low parts, same accumulator)
                                    const uint64_t bl = smem_desc(pbase + (K::OFF_PLO - K::OFF_P) + pg * 256, 128, 16 * 128);
                                    mma_bf16(ocol, a, bl, idPV, 1u);
                                }
                            }
                        }
                    }
                    mma_commit(bar(B::PEMPTY + t % NSB));
                    mma_commit(bar(B::VEMPTY + vs));
                    if (t0 + kTP >= it.npg) mma_commit(bar(B::ODONE + (pc & 1)));
                }
                ++pc;
                if (ok) it.advance(p);
            }
            mma_commit(bar(B::DONE + 1));
            wait_bar(bar(B::DONE + 1), 0, drain);
        }
        __syncwarp();
    } else if (warp == kMergeWarp) {
        // ------------------------------------------------------------ hand-offs and the last piece's pre-merge
        // The split pieces before the CTA's last piece come here in order (the
        // softmax warps store a partial; this warp reads the segment's ticket:
        // when every other piece is published it merges at once, else it makes
        // the partial visible GPU-wide, draws a ticket and merges if that ticket
        // is the last).  Then, when the last piece is split and ends its
        // segment, this warp waits for the segment's earlier pieces to be
        // published and merges them into shared memory, so that the last
        // epilogue only adds its own part.
        griddep_wait();                   // tickets and partials of the previous launch are settled
        int n_expect = 0;
        PieceIter<CASC> w = it;                 // -> the last piece
        for (;;) {
            PieceIter<CASC> nx = w;
            nx.advance(p);
            if (!nx.valid()) break;
            if (w.S0 < u0 || w.S1 > u1) ++n_expect;
            w = nx;
        }
        int* mq = reinterpret_cast<int*>(smem + K::OFF_MQ);
        bool ok = true;
        for (int n = 0; n < n_expect; ++n) {
            bool wv = lane == 0 ? wait_bar(bar(B::MQFULL + (n & 3)), (n >> 2) & 1, ctl) : true;
            if (!(ok = __shfl_sync(0xffffffffu, wv, 0))) break;
            __syncwarp();
            const int* task = mq + (n & 3) * 8;
            const int seg_b = task[0], hg = task[1], S0 = task[4], S1 = task[5];
            int last = 0;
            if (lane == 0) {
                const int need = part.owner(S1 - 1) - part.owner(S0) + 1;
                int* ticket = p.tickets + seg_b * p.num_kv_heads + hg;
                if (ld_acquire_gpu(ticket) == need - 1) {
                    // every other piece is published (and visible): merge without publishing this one
                    last = 1;
                } else {
                    // publish the partial (stored before the arrive) and draw the ticket
                    last = atom_add_acq_rel_gpu(ticket, 1) == need - 1;
                }
                if (last) *ticket = 0;                  // ready for the next launch
            }
            last = __shfl_sync(0xffffffffu, last, 0);
            __syncwarp();
            if (last) merge_segment_warp<D, CASC>(p, hg, task[2], task[3], S0, S1, part, lane, task[6]);
        }
        if constexpr (SPLIT) {
            if (ok && w.S0 < u0 && w.S1 <= u1) {
                const int c_first = part.owner(w.S0);          // this CTA is the segment's last
                int* ticket = p.tickets + w.cur.b * Hkv + w.hg;
                const int ncol = HG * G * w.cur.Q;
                const uint64_t t0 = globaltimer_ns();
                // (relaxed polls, one acquire fence once the count is reached: an acquire
                // per poll would slow the rest of the SM)
                while (*gstate == 0 && !*abort_flag && globaltimer_ns() - t0 < p.wait_limit_ns) {
                    int v = 0;
                    if (lane == 0) {
                        v = ld_relaxed_gpu(ticket);
                        if (v == cta - c_first) fence_acquire_gpu();
                    }
                    v = __shfl_sync(0xffffffffu, v, 0);
                    if (v == cta - c_first) {
                        int claimed = 0;
                        if (lane == 0) claimed = atomicCAS(const_cast<int*>(gstate), 0, 1) == 0;
                        claimed = __shfl_sync(0xffffffffu, claimed, 0);
                        __syncwarp();
                        if (claimed) {
                            // the earlier pieces in CTA order, the same steps as merge_segment_warp
                            constexpr int DPL = D / 32;
                            float M[RMAX], den[RMAX], num[RMAX][DPL];
#pragma unroll
                            for (int k = 0; k < RMAX; ++k) {
                                M[k] = -INFINITY;
                                den[k] = 0.f;
#pragma unroll
                                for (int x = 0; x < DPL; ++x) num[k][x] = 0.f;
                            }
                            for (int c = c_first; c < cta; ++c) {
                                const float* sl = slot_ptr(p, c, w.S0, part.start(c));
#pragma unroll
                                for (int k = 0; k < RMAX; ++k) {
                                    const bool ld = k < ncol;
                                    const float m = ld ? __ldcg(sl + k) : -INFINITY;
                                    const float l = ld ? __ldcg(sl + p.rows_pad + k) : 0.f;
                                    float wo, wn;
                                    merge_weights(M[k], m, wo, wn);
                                    den[k] = merge_acc(den[k], wo, l, wn);
#pragma unroll
                                    for (int x = 0; x < DPL; ++x) {
                                        const float a = ld ? __ldcg(sl + 2 * p.rows_pad + (size_t)k * D + lane + 32 * x) : 0.f;
                                        num[k][x] = merge_acc(num[k][x], wo, a, wn);
                                    }
                                }
                            }
#pragma unroll
                            for (int k = 0; k < RMAX; ++k) {
                                if (lane == 0) {
                                    gbuf[k] = M[k];
                                    gbuf[RMAX + k] = den[k];
                                }
#pragma unroll
                                for (int x = 0; x < DPL; ++x) gbuf[2 * RMAX + k * D + lane + 32 * x] = num[k][x];
                            }
                            __threadfence_block();
                            __syncwarp();
                            if (lane == 0) {
                                *ticket = 0;                    // ready for the next launch
                                *gstate = 2;
                            }
                        }
                        break;
                    }
                    __nanosleep(1000);
                }
            }
        }
        __syncwarp();
    } else if (warp < 4) {
        // ------------------------------------------------------------ softmax / rescale
        // One thread per token row of S^T (TMEM lane).  At a piece's end its
        // column sums and reference max go to lred / emref (double-buffered by
        // piece parity); the piece's epilogue then runs in the epilogue
        // warpgroup (EWG), or here after the next piece's first tile.
        const int tt = tid;
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        float* red = reinterpret_cast<float*>(smem + K::OFF_RED);
        int t = 0, pc = 0, jt = 0;
        bool aborted = false;
        float m_ref[RMAX], l_part[RMAX];
        bool pend = false;                   // (without EWG) the finished piece whose epilogue is pending
        PieceDesc pd{};
#pragma unroll
        for (int n = 0; n < RMAX; ++n) {
            m_ref[n] = -INFINITY;
            l_part[n] = 0.f;
        }
        bool in_piece = it.valid();

        for (;;) {
            if (in_piece) {
                const int Q = it.cur.Q, R = G * Q, L = it.cur.L, lim0 = L - Q;
                const int np = min(kTP, it.npg - jt * kTP);
                const int vs = t % NSV;
                const uint32_t obase = K::COL_O + (pc & 1) * K::HGMAX * K::NM;
                // this thread's token: unit slot k of the tile -> (page, kv-head), position
                const int k = tt >> 4;
                const int qu = it.pg0 + jt * kTP + k;
                const int qpg = div_small(qu, HG);
                const int hh = qu - qpg * HG;
                const int pos = ((CASC ? it.cur.pb : 0) + qpg) * kBlock + (tt & 15);
                const bool tok_ok = k < np && pos < L;
                // visible columns: [lo, hi) of this head's R rows (causal within the window)
                const int lo = hh * R + ((CASC && p.cascade == 1) ? 0 : max(0, pos - lim0) * G), hi = hh * R + R;

                bool okw = wait_bar(bar(B::SFULL + t % NSB), (t / NSB) & 1, ctl);
                // (FP8) this token's page scales and the columns' factors: S^T holds
                // (2^E_n q_n) . code split over columns n and 8 + n, and V enters as codes
                float kscale = 1.f, vscale = 1.f, cf[FP8 ? RMAX : 1];
                if constexpr (FP8) {
                    okw = wait_bar(bar(B::SCALE + t % K::NSC), (t / K::NSC) & 1, ctl) && okw;
                    const float* sc = reinterpret_cast<const float*>(smem + K::OFF_SC) + (t % K::NSC) * 32;
                    kscale = sc[k];
                    vscale = sc[8 + k];
                    // P carries the v scale into fp16 operands: P < 2^8 keeps P * vscale finite for
                    // scales up to 255 (|v| below ~114,000 before encoding)
                    if (vscale > 255.f) raise_error(p.err, PKV_DEVERR_RANGE);
#pragma unroll
                    for (int n = 0; n < RMAX; ++n) cf[n] = sc[16 + n] * (p.scale_log2 * kscale);
                }
                tc_fence_after();
                float s[RMAX];
#pragma unroll
                for (int c = 0; c < RMAX; c += 16) {
                    float tmp[16];
                    tmem_ld16(tmem + lane_base + K::COL_S + (t % NSB) * K::NM + c, tmp);
                    if constexpr (FP8 && RMAX > 8) {
                        // hi + lo q terms: columns c + x and RMAX + c + x
                        float tl[16];
                        tmem_ld16(tmem + lane_base + K::COL_S + (t % NSB) * K::NM + RMAX + c, tl);
#pragma unroll
                        for (int x = 0; x < 16 && c + x < RMAX; ++x) s[c + x] = tmp[x] + tl[x];
                    } else {
#pragma unroll
                        for (int x = 0; x < 16 && c + x < RMAX; ++x) {
                            if constexpr (FP8)
                                s[c + x] = tmp[x] + tmp[x + RMAX];   // hi + lo q terms (RMAX = 8)
                            else
                                s[c + x] = tmp[x];
                        }
                    }
                }
                bool need = false;
#pragma unroll
                for (int n = 0; n < RMAX; ++n) {
                    const bool vis = tok_ok && n >= lo && n < hi;
                    if constexpr (FP8)
                        s[n] = vis ? s[n] * cf[n] : -INFINITY;
                    else
                        s[n] = vis ? s[n] * p.scale_log2 : -INFINITY;
                    need |= s[n] > m_ref[n] + kRescaleSlack;
                }
                // The FP8 kernel votes without blocking: each warp posts its vote and arrives on
                // the tile's vote barrier, P is computed against the current reference meanwhile,
                // and only then is the vote read (a raise recomputes P).  A vote barrier that
                // timed out counts as a raise, whose first barrier then winds all warps down.
                // (The bf16 kernels measured no faster this way: they keep the blocking vote.)
                constexpr bool kSpec = SPLIT && FP8;
                float pr[RMAX];
                bool raise;
                if constexpr (kSpec) {
                    int* vote = reinterpret_cast<int*>(smem + K::OFF_VOTE) + (t & 1) * 4;
                    const bool wneed = __any_sync(0xffffffffu, need || !okw);
                    if (lane == 0) {
                        vote[warp] = wneed ? 1 : 0;
                        mbar_arrive(bar(B::VOTE + (t & 1)));
                    }
#pragma unroll
                    for (int n = 0; n < RMAX; ++n) pr[n] = (s[n] == -INFINITY) ? 0.f : fast_exp2(s[n] - m_ref[n]);
                    const bool okv = wait_bar(bar(B::VOTE + (t & 1)), (t >> 1) & 1, ctl);
                    const volatile int* vq = vote;
                    raise = !okv || (vq[0] | vq[1] | vq[2] | vq[3]) != 0;
                } else {
                    raise = bar_red_or(kBarSoft, kSoftThreads, need || !okw);
                }
                if (raise) {
                    // raise the reference to this tile's max (first tile of a piece, or a big jump):
                    // per (unit slot, column) maxima over the slot's 16 tokens, then per column
                    if constexpr (RMAX <= 16) {
                        float a[RMAX];
#pragma unroll
                        for (int n = 0; n < RMAX; ++n) a[n] = s[n];
                        int col = 0;
                        Butterfly<RMAX, 8, true>::run(a, lane, col);
                        if ((lane & (16 / RMAX - 1)) == 0) red[k * RMAX + col] = a[0];
                    } else {
#pragma unroll
                        for (int n = 0; n < RMAX; ++n) {
                            float mx = s[n];
#pragma unroll
                            for (int o = 8; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                            if ((tt & 15) == 0) red[k * RMAX + n] = mx;
                        }
                    }
                    if (bar_red_or(kBarSoft, kSoftThreads, !okw || *abort_flag)) {
                        aborted = true;
                        break;
                    }
                    float alpha[RMAX];
                    bool any_scale = false;
#pragma unroll
                    for (int n = 0; n < RMAX; ++n) {
                        float tm = -INFINITY;
#pragma unroll
                        for (int kk = 0; kk < kTP; ++kk) tm = fmaxf(tm, red[kk * RMAX + n]);
                        const float mn = fmaxf(m_ref[n], tm);
                        alpha[n] = (m_ref[n] == -INFINITY) ? 0.f : fast_exp2(m_ref[n] - mn);
                        any_scale |= (alpha[n] != 1.f) && (m_ref[n] != -INFINITY);
                        m_ref[n] = mn;
                        l_part[n] *= alpha[n];
                    }
                    if (jt > 0 && any_scale) {
                        // O^T (TMEM) *= alpha once the previous tile's P.V has landed, in the
                        // accumulator of every kv-head of the segment
                        wait_bar(bar(B::PEMPTY + (t - 1) % NSB), ((t - 1) / NSB) & 1, ctl);
                        tc_fence_after();
                        for (int h2 = 0; h2 < HG; ++h2) {
#pragma unroll
                            for (int c = 0; c < K::NM; c += 16) {
                                float o[16];
                                tmem_ld16(tmem + lane_base + obase + h2 * K::NM + c, o);
#pragma unroll
                                for (int x = 0; x < 16; ++x) {
                                    const int n = SPLIT ? (c + x) / 2 : (c + x);
                                    o[x] *= n < RMAX ? alpha[n] : 1.f;
                                }
                                tmem_st16(tmem + lane_base + obase + h2 * K::NM + c, o);
                            }
                        }
                    }
                    // keep red[] stable until every thread has read it
                    named_bar_sync(kBarSoft, kSoftThreads);
                }
                if (!kSpec || raise) {
#pragma unroll
                    for (int n = 0; n < RMAX; ++n) pr[n] = (s[n] == -INFINITY) ? 0.f : fast_exp2(s[n] - m_ref[n]);
                }
#pragma unroll
                for (int n = 0; n < RMAX; ++n) l_part[n] += pr[n];
                // P buffer t % NSB is free once the P.V of tile t - NSB has completed
                if (t >= NSB) wait_bar(bar(B::PEMPTY + t % NSB), ((t / NSB) - 1) & 1, ctl);
                uint8_t* pdst = smem + K::OFF_P + (t % NSB) * K::PBUF + tt * 16;
#pragma unroll
                for (int cc = 0; cc < (NPAD + 7) / 8; ++cc) {      // (a last group past RMAX is 0)
                    uint32_t w4[4], l4[4];
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        float a, b;
                        if constexpr (SPLIT) {
                            const int n = cc * 4 + h;          // physical columns 2n (high) and 2n+1 (low)
                            const float pv = FP8 ? pr[n] * vscale : pr[n];
                            // (FP8: fp16 parts, the type of the widened V)
                            const float hi = FP8 ? __half2float(__float2half_rn(pv)) : __bfloat162float(__float2bfloat16_rn(pv));
                            a = hi;
                            b = pv - hi;
                        } else {
                            // wide: column n's high part here, its low part in the second ring
                            const int n0 = cc * 8 + 2 * h;
                            a = n0 < RMAX ? (FP8 ? pr[n0] * vscale : pr[n0]) : 0.f;
                            b = n0 + 1 < RMAX ? (FP8 ? pr[n0 + 1] * vscale : pr[n0 + 1]) : 0.f;
                            const float ah = FP8 ? __half2float(__float2half_rn(a)) : __bfloat162float(__float2bfloat16_rn(a));
                            const float bh = FP8 ? __half2float(__float2half_rn(b)) : __bfloat162float(__float2bfloat16_rn(b));
                            l4[h] = FP8 ? pack_f16x2(a - ah, b - bh) : pack_bf16x2(a - ah, b - bh);
                            a = ah;
                            b = bh;
                        }
                        w4[h] = FP8 ? pack_f16x2(a, b) : pack_bf16x2(a, b);
                    }
                    *reinterpret_cast<uint4*>(pdst + cc * (16 * 128)) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                    if constexpr (!SPLIT)
                        *reinterpret_cast<uint4*>(pdst + (K::OFF_PLO - K::OFF_P) + cc * (16 * 128)) =
                            make_uint4(l4[0], l4[1], l4[2], l4[3]);
                }
                if constexpr (FP8) {
                    // this warpgroup widens V(t) (it has time to spare between tiles; the epilogue
                    // warpgroup keeps the piece epilogues): every thread acquires the landed pages
                    wait_bar(bar(B::VLAND + vs), (t / NSV) & 1, ctl);
                    widen(smem + K::OFF_V + vs * (K::TILE + K::VSLACK), tt, kBarSoft);
                    mbar_arrive(bar(B::VFULL + vs));
                }
                // unwritten tail slots of the sequence's last page: zero their V rows (they may hold NaN)
                if (k < np && pos >= L) {
                    wait_bar(bar(B::VFULL + vs), (t / NSV) & 1, ctl);
                    uint8_t* vrow = smem + K::OFF_V + vs * (K::TILE + K::VSLACK) + k * K::PAGE +
                                    ((tt & 15) >> 3) * (K::NCH * 128) + (tt & 7) * 16;
#pragma unroll
                    for (int c = 0; c < K::NCH; ++c) *reinterpret_cast<uint4*>(vrow + c * 128) = make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(bar(B::PFULL + t % NSB));

                ++t;
            }
            if constexpr (!EWG) {
                if (pend && (!in_piece || jt == 0)) {
                    pend = false;
                    pd.last = !in_piece;
                    piece_epilogue(pd, tt, kBarSoft);
                }
            }
            if (!in_piece) break;

            if (++jt * kTP >= it.npg) {
                // piece end: its column sums and reference max for the epilogue
                const int par = pc & 1;
                if (EWG && pc >= 2) {
                    // lred / emref of this parity are free once piece pc - 2's epilogue has read them
                    const bool okf = wait_bar(bar(B::OFREE + par), ((pc >> 1) - 1) & 1, ctl);
                    if (bar_red_or(kBarSoft, kSoftThreads, !okf)) {
                        aborted = true;
                        break;
                    }
                }
                float* lw = lred + (par * 4 + warp) * RMAX;
                {
                    // (a power-of-two width for the butterfly: RMAX = 24 is padded to 32)
                    constexpr int RB = RMAX <= 8 ? 8 : RMAX <= 16 ? 16 : 32;
                    float lb[RB];
#pragma unroll
                    for (int n = 0; n < RB; ++n) lb[n] = n < RMAX ? l_part[n] : 0.f;
                    int col = 0;
                    Butterfly<RB, 16, false>::run(lb, lane, col);
                    if ((lane & (32 / RB - 1)) == 0 && col < RMAX) lw[col] = lb[0];
                }
#pragma unroll
                for (int n = 0; n < RMAX; ++n)
                    if (tt == 0) emref[par * RMAX + n] = m_ref[n];
                pd.b = it.cur.b;
                pd.hg = it.hg;
                pd.qoff = it.cur.qoff;
                pd.Q = it.cur.Q;
                pd.S0 = it.S0;
                pd.S1 = it.S1;
                pd.pc = pc;
                pd.pb = it.cur.pb;
#pragma unroll
                for (int n = 0; n < RMAX; ++n) {
                    m_ref[n] = -INFINITY;
                    l_part[n] = 0.f;
                }
                ++pc;
                jt = 0;
                it.advance(p);
                in_piece = it.valid();
                if constexpr (EWG) {
                    // hand the piece over: descriptor, then every thread's arrive (its sums are stored)
                    if (tt == 0) {
                        int* q = pdesc + par * 8;
                        q[0] = pd.b;
                        q[1] = pd.hg;
                        q[2] = pd.qoff;
                        q[3] = pd.Q;
                        q[4] = pd.S0;
                        q[5] = pd.S1;
                        q[6] = in_piece ? 0 : 1;
                        q[7] = pd.pb;
                    }
                    mbar_arrive(bar(B::PREADY + par));
                } else {
                    pend = true;
                }
            }
        }
        (void)aborted;
    } else if (warp >= kEpiWarp0) {
        // ------------------------------------------------------------ epilogue warpgroup
        if constexpr (EWG) {
            const int tt = tid - kEpiWarp0 * 32;
            auto take_piece = [&](int pc) -> PieceDesc {
                const int* q = pdesc + (pc & 1) * 8;
                PieceDesc d;
                d.b = q[0];
                d.hg = q[1];
                d.qoff = q[2];
                d.Q = q[3];
                d.S0 = q[4];
                d.S1 = q[5];
                d.last = q[6] != 0;
                d.pb = q[7];
                d.pc = pc;
                return d;
            };
            for (int pc = 0;; ++pc) {
                const bool okr = wait_bar(bar(B::PREADY + (pc & 1)), (pc >> 1) & 1, ctl);
                if (bar_red_or(kBarEpi, kSoftThreads, !okr)) break;
                const PieceDesc d = take_piece(pc);
                piece_epilogue(d, tt, kBarEpi);
                if (d.last) break;
            }
        }
    }

    // ---------------------------------------------------------------- teardown
    // (every role reaches this barrier from its own code path: the non-.aligned form)
    tc_fence_before();
    cta_bar_sync();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, K::TMEM_COLS);
    }
}

template <int D, int NPAD, bool SPLIT, int NSK, int NSV, bool EWG, bool FP8 = false, bool CASC = false>
static cudaError_t launch_t(const AttnParams& p, int ncta, cudaStream_t st) {
    using K = Cfg<D, NPAD, SPLIT, NSK, NSV, EWG, FP8>;
    static std::atomic<uint64_t> attr_set{0};
    return launch_pdl_bigsmem(attr_set, attn_tc_kernel<D, NPAD, SPLIT, NSK, NSV, EWG, FP8, CASC>, dim3(ncta),
                              dim3(threads_of<EWG>()), (size_t)K::SMEM, st, p);
}

}  // namespace tc

// Columns per segment for the tensor-core kernel: up to 8 (with the bf16
// high/low split of P, N = 16) when the rows of one kv-head fit, else up to 32.
static int tc_col_limit(int rows) { return rows <= 8 ? 8 : 32; }

// kv-heads per segment: the largest divisor of Hkv whose columns
// (heads x G x max_q_len) fit the column limit.
// At most 4 (narrow) or 2 (wide): each kv-head of a segment has its own O^T
// accumulator in TMEM.
int tc_heads_per_segment(int num_kv_heads, int rows, bool fp8) {
    // (FP8 wide segments: 16 columns, each q row split over two)
    const int lim = fp8 && rows > 8 ? 16 : tc_col_limit(rows), cap = rows <= 8 ? 4 : 2;
    int hg = 1;
    for (int h = 1; h <= min(num_kv_heads, cap); ++h)
        if (num_kv_heads % h == 0 && h * rows <= lim) hg = h;
    return hg;
}

// bf16 cache, head_dim 64/128, R = G * max_q_len <= 32; FP8 cache, head_dim
// 64/128, R <= 8.  Narrow segments (N = 16) run the epilogue in its own
// warpgroup; wide ones (N = 32), whose softmax needs more registers than a
// 384-thread block leaves, in the softmax warps.  Wide head_dim 128 segments
// of at most 20 or 24 columns (a 5-token verify window at G = 4: 20) take a
// kernel whose softmax and epilogue handle only those of the 32 MMA columns;
// the 20-column softmax fits a 384-thread block, so that one has the epilogue
// warpgroup too.
cudaError_t launch_attention_tc(const AttnParams& p, int head_dim, bool fp8, int ncta, cudaStream_t st) {
    const bool split = tc_col_limit(p.rows) == 8;
    if (p.cascade != 0) {                      // (bf16 caches only: the host checks)
        if (fp8) return cudaErrorInvalidValue;
        if (head_dim == 128)
            return split ? tc::launch_t<128, 16, true, 2, 4, true, false, true>(p, ncta, st)
                         : tc::launch_t<128, 32, false, 2, 2, false, false, true>(p, ncta, st);
        return split ? tc::launch_t<64, 16, true, 4, 6, true, false, true>(p, ncta, st)
                     : tc::launch_t<64, 32, false, 4, 4, false, false, true>(p, ncta, st);
    }
    if (head_dim == 128)
        return fp8 && split ? tc::launch_t<128, 16, true, 4, 4, true, true>(p, ncta, st)
               : fp8        ? tc::launch_t<128, 32, false, 2, 3, true, true>(p, ncta, st)
               : split      ? tc::launch_t<128, 16, true, 2, 4, true>(p, ncta, st)
               : p.hg * p.rows <= 20 ? tc::launch_t<128, 20, false, 2, 2, true>(p, ncta, st)
               : p.hg * p.rows <= 24 ? tc::launch_t<128, 24, false, 2, 2, false>(p, ncta, st)
                                     : tc::launch_t<128, 32, false, 2, 2, false>(p, ncta, st);
    return fp8     ? tc::launch_t<64, 16, true, 6, 8, true, true>(p, ncta, st)
           : split ? tc::launch_t<64, 16, true, 4, 6, true>(p, ncta, st)
                   : tc::launch_t<64, 32, false, 4, 4, false>(p, ncta, st);
}

}  // namespace pkv
