// Shared device helpers of libpagedkv: number formats, the balanced work
// partition over (sequence, kv-head, page) units and the split merge.
//
// Work partition ("Split-K" of the lfm25-inference README's paged GQA/XQA
// decode attention, restated for a persistent grid).  Every (sequence b,
// kv-head g) pair is a segment of ceil(L_b / 16) page units; segments are
// laid end to end in (b, g) order and the W units are cut into P equal
// ranges, one per CTA: CTA c owns units [floor(c W / P), floor((c+1) W / P)).
// A segment that falls inside one CTA is finished there; a segment cut by a
// range boundary leaves one partial (m, l, acc) per CTA it touches, and the
// CTA that finishes last (a ticket per segment, no waiting) merges them in
// CTA order.  The cut depends on lengths only, never on physical block ids.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/pagedkv.h"

namespace pkv {

constexpr int kBlock = 16;                 // tokens per page (block_size)
constexpr float kLog2e = 1.4426950408889634f;

// ------------------------------------------------------------------ formats

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Two E4M3 codes (low byte = first element) -> two floats, exact.
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t two_codes) {
    __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(two_codes & 0xffffu), __NV_E4M3);
    __half2 hh = *reinterpret_cast<__half2*>(&h);
    return __half22float2(hh);
}

__device__ __forceinline__ void raise_error(int* err, int bits) {
    if (err) atomicOr(err, bits);
}

// Programmatic dependent launch: a kernel launched with
// programmaticStreamSerialization may start while the previous kernel on the
// stream runs; griddep_wait() blocks until that kernel has completed and its
// memory is visible (a no-op for a normal launch).  griddep_launch() lets the
// next kernel on the stream start early.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }

template <typename... Args>
__host__ inline cudaError_t launch_pdl(void (*kern)(Args...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                                       Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

// launch_pdl for a kernel with more than 48 KiB of dynamic shared memory.
// The function attribute that allows it is set once per device (`done` holds
// one bit per device, static in the caller, one per kernel): setting it on
// every launch costs a driver call for nothing.  A launch refused after the
// attribute was lost (a device reset) sets it again and retries once.
template <typename... Args>
__host__ inline cudaError_t launch_pdl_bigsmem(std::atomic<uint64_t>& done, void (*kern)(Args...), dim3 grid,
                                               dim3 block, size_t smem, cudaStream_t st, Args... args) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev < 64 ? (1ull << dev) : 0ull;
    const bool set = bit != 0 && (done.load(std::memory_order_acquire) & bit) != 0;
    if (!set) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        if (bit) done.fetch_or(bit, std::memory_order_release);
    }
    e = launch_pdl(kern, grid, block, smem, st, args...);
    if (e != cudaSuccess && set) {
        (void)cudaGetLastError();
        done.fetch_and(~bit, std::memory_order_release);
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        done.fetch_or(bit, std::memory_order_release);
        e = launch_pdl(kern, grid, block, smem, st, args...);
    }
    return e;
}

// ------------------------------------------------------------------ workspace

struct WorkspaceLayout {
    size_t tickets_off;     // int32 [num_seqs * Hkv]
    size_t partials_off;    // float [num_ctas][2][slot_floats]
    size_t slot_floats;     // rows_pad * (head_dim + 2)
    size_t total;
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

__host__ inline WorkspaceLayout workspace_layout(int num_seqs, int num_kv_heads, int head_dim,
                                                 int rows_pad, int num_ctas) {
    WorkspaceLayout w;
    w.tickets_off = 256;
    w.partials_off = align_up(w.tickets_off + sizeof(int32_t) * (size_t)num_seqs * num_kv_heads, 256);
    w.slot_floats = (size_t)rows_pad * (head_dim + 2);
    w.total = w.partials_off + sizeof(float) * w.slot_floats * 2 * (size_t)num_ctas;
    return w;
}

// ------------------------------------------------------------------ parameters

struct AttnParams {
    const uint8_t* k_cache;
    const uint8_t* v_cache;
    const float* k_scales;
    const float* v_scales;
    const __nv_bfloat16* q;
    __nv_bfloat16* out;
    const int32_t* block_tables;
    const int32_t* context_lens;
    const int32_t* q_lens;
    int* err;                  // workspace error word
    int* tickets;              // workspace tickets
    float* partials;           // workspace partial slots
    int64_t num_blocks;
    int num_seqs;
    int num_q_heads;
    int num_kv_heads;
    int group;                 // Hq / Hkv
    int max_blocks_per_seq;
    int max_q_len;             // host bound on q_lens
    int rows;                  // group * max_q_len (rows of the widest segment)
    int rows_pad;              // slot row capacity
    int slot_floats;
    float scale_log2;          // scale * log2(e)
    int hg;                    // kv-heads per segment (tensor-core kernel; 1 elsewhere)
    uint64_t wait_limit_ns;    // every bounded wait of the tensor-core kernel gives up after this
    const int* hold;           // tests of the timeout path only: wait for *hold != 0 first (nullptr: no wait)
    // num_kv_heads and group above count virtual kv-heads: when a kv-head's
    // query rows (G * max_q_len) exceed the 32 columns a segment holds, its G
    // query heads are split into kv_split consecutive groups, each a virtual
    // kv-head (so query head h still reads virtual head h / group) that reads
    // the pages of cache kv-head (virtual head) / kv_split.
    int kv_split;
    int cache_kv_heads;        // kv-heads of the cache (num_kv_heads / kv_split)
    // Shared-prefix cascade (pkv_paged_attention_cascade).  0: plain call.
    // 1, the prefix pass: "sequence" g is group g = sequences
    //    [group_starts[g], group_starts[g + 1]), context_lens holds the groups'
    //    shared prefix lengths, its query window is all the group's q rows
    //    (consecutive in q), its block-table row is its first sequence's, no
    //    causal mask (every row sees the whole prefix), and the results go to
    //    state_o / state_lse instead of out.
    // 2, the suffix pass: a sequence's pages start after its group's prefix,
    //    and its rows are merged with the prefix pass's states before out.
    int cascade;
    const int32_t* group_starts;       // [num_groups + 1]
    const int32_t* group_prefix_lens;  // [num_groups] (suffix pass)
    int num_groups;
    int num_seqs_total;                // sequences of the batch (the prefix pass's num_seqs counts groups)
    float* state_o;                    // [rows][Hq][D] fp32: normalised output of the prefix pass
    float* state_lse;                  // [rows][Hq] fp32: its log2-sum-exp (scale * log2 e units)
};

// Virtual kv-heads per cache kv-head: the smallest divisor of the GQA group
// that leaves at most `limit` query rows per virtual head (32 for bf16 caches;
// for FP8 caches the rows of the FP8 tensor-core kernel: 16 at head_dim 128,
// 8 at 64 for windows of up to 8 tokens; each virtual head's segment re-reads
// the cache kv-head's pages, mostly from L2, which still beats the CUDA-core
// kernel severalfold).
__host__ inline int kv_split_for(int group, int max_q_len, int limit = 32) {
    for (int ks = 1; ks < group; ++ks)
        if (group % ks == 0 && (group / ks) * max_q_len <= limit) return ks;
    return group;
}
__host__ inline int kv_split_limit(bool fp8, int head_dim, int max_q_len) {
    return !fp8 ? 32 : head_dim == 128 ? 16 : max_q_len <= 8 ? 8 : 32;
}

// Cache kv-head of virtual kv-head vh.
__device__ __forceinline__ int cache_head(const AttnParams& p, int vh);

// The wait limit and hold flag of the next launches (pkv_debug_set_wait_limit),
// copied into AttnParams by both attention entry points.
void fill_debug(AttnParams& p);

// Kernel choice and grid of one attention call (see plan_attention in api.cu).
struct AttnLaunch {
    bool tc;        // tensor-core kernel
    int ncta;       // grid size
    int rows_pad;   // partial-slot rows
    int hg;         // kv-heads per segment
};

// ------------------------------------------------------------------ planning

// floor(num / den) for 0 <= num < 2^47 and 0 < den < 2^31 with a quotient
// below 2^31, without a 64-bit division: a float estimate (relative error near
// 2^-22), a second estimate on the remainder (now within one of the quotient)
// and one exact integer correction step.
__device__ __forceinline__ int floor_div_small(long long num, int den) {
    int q = (int)__fdividef((float)num, (float)den);
    long long r = num - (long long)q * den;
    q += (int)__fdividef((float)r, (float)den);
    r = num - (long long)q * den;
    if (r < 0) --q;
    else if (r >= den) ++q;
    return q;
}

// floor(n / d) for 0 <= n < 2^20 and d >= 1 by one approximate float
// division: the quotient of n + 1/2 lies at least 1 / (2 d) from an integer,
// and the division's relative error (a few units of 2^-24) keeps it on the
// right side for numerators this small.
__device__ __forceinline__ int div_small(int n, int d) {
    return (int)__fdividef((float)n + 0.5f, (float)d);
}

__device__ __forceinline__ int cache_head(const AttnParams& p, int vh) {
    return p.kv_split == 1 ? vh : div_small(vh, p.kv_split);
}

// CTAs that take part: enough that every one gets at least kMinUnitsPerCta
// units (two 128-token tiles), so a small batch is not spread so thin that a
// segment crosses dozens of CTAs and its merge walks dozens of partials; but
// at least one per non-empty segment (S of them), so short segments are not
// packed several to a CTA, whose piece epilogues would then run one after
// another.
constexpr int kMinUnitsPerCta = 16;
__device__ __forceinline__ int participating_ctas(int ncta, int W, int S) {
    return W <= 0 ? 0 : max(1, min(ncta, max(W / kMinUnitsPerCta, S)));
}

// CTA owning unit u under the partition above (P = participating CTAs <= W,
// so every CTA in [owner(S0), owner(S1 - 1)] holds a piece of [S0, S1)).
__device__ __forceinline__ int owner_cta(int u, int W, int ncta) {
    return floor_div_small((long long)(u + 1) * ncta - 1, W);
}
// First unit of CTA c, floor(c W / P).
__device__ __forceinline__ int cta_start(int c, int W, int ncta) {
    return floor_div_small((long long)c * W, ncta);
}

// The partition a launch uses: CTA c streams units [start(c), start(c + 1)).
// Either the equal split of the W units over P CTAs (the formulas above), or
// a table of P + 1 boundaries in shared memory (bnd != nullptr) cut so that
// every CTA gets an equal share of units plus a fixed cost per segment piece.
// Every CTA holds the same table, so owner() and start() agree across CTAs.
struct Part {
    int W, P;
    const int* bnd;
    __device__ __forceinline__ int start(int c) const { return bnd ? bnd[c] : cta_start(c, W, P); }
    // the CTA whose range holds unit u (u < W): the last c with start(c) <= u
    __device__ __forceinline__ int owner(int u) const {
        if (!bnd) return owner_cta(u, W, P);
        int lo = 0, hi = P - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (bnd[mid] <= u) lo = mid;
            else hi = mid - 1;
        }
        return lo;
    }
};

// A sequence's length, query rows and first page (pages before it belong to
// its group's shared prefix, attended by the cascade's prefix pass).
struct SeqInfo {
    int L, Q, pb;
};
// CASC: compiled for a kernel that a cascade launches (else p.cascade is 0
// and none of its code is there).
template <bool CASC = false>
__device__ __forceinline__ SeqInfo seq_info(const AttnParams& p, int b) {
    SeqInfo r{p.context_lens[b], 0, 0};
    if constexpr (!CASC) {
        r.Q = p.q_lens[b];
        return r;
    }
    if (p.cascade == 1) {
        const int s0 = max(0, p.group_starts[b]), e = min(p.group_starts[b + 1], p.num_seqs_total);
        for (int s = s0; s < e; ++s) r.Q += p.q_lens[s];
        if (p.group_starts[b] < 0 || p.group_starts[b] >= p.num_seqs_total) r.Q = 0;   // (no rows to read)
        return r;
    }
    r.Q = p.q_lens[b];
    if (p.cascade == 2) {            // the group holding b: the last g with group_starts[g] <= b
        int lo = 0, hi = p.num_groups - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (p.group_starts[mid] <= b) lo = mid;
            else hi = mid - 1;
        }
        r.pb = p.group_prefix_lens[lo] / kBlock;
    }
    return r;
}

// Units (pages x kv-heads) of sequence b; sequences with no query rows or
// invalid lengths (Q > L, Q above the launch's max_q_len, more pages than a
// block-table row holds, a group prefix reaching into the query window)
// contribute none.  In the prefix pass a group with no prefix has no units
// and is not an error.
template <bool CASC = false>
__device__ __forceinline__ bool seq_valid(const AttnParams& p, int L, int Q, int pb) {
    const bool fits = Q > 0 && Q <= p.max_q_len && (L + kBlock - 1) / kBlock <= p.max_blocks_per_seq;
    if constexpr (!CASC) return fits && Q <= L;
    if (p.cascade == 1) return fits && L > 0 && L % kBlock == 0;     // (prefixes are whole blocks)
    return fits && Q <= L && pb * kBlock <= L - Q;
}
template <bool CASC = false>
__device__ __forceinline__ bool seq_error(const AttnParams& p, int L, int Q, int pb) {
    if (CASC && p.cascade == 1) return L != 0 && !seq_valid<CASC>(p, L, Q, pb);
    return Q != 0 && !seq_valid<CASC>(p, L, Q, pb);
}
template <bool CASC = false>
__device__ __forceinline__ int seq_units(const AttnParams& p, int L, int Q, int pb) {
    return seq_valid<CASC>(p, L, Q, pb) ? ((L + kBlock - 1) / kBlock - (CASC ? pb : 0)) * p.num_kv_heads : 0;
}
// q rows of sequence b in the packed q / out tensors.
__device__ __forceinline__ int seq_qrows(int Q) { return Q > 0 ? Q : 0; }

struct Cursor {
    int b;          // current sequence
    int Ub;         // units before sequence b
    int qoff;       // first q row of sequence b
    int L, Q, nb;   // its context length, query length, pages it attends (from page pb on)
    int pb;         // its first page (0 unless a cascade's suffix pass)
};

// Block-wide inclusive scan of one int per thread (NT threads, NT % 32 == 0).
template <int NT>
__device__ __forceinline__ int block_scan_incl(int v, int* scratch /* NT/32 + 1 ints */) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    if (lane == 31) scratch[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int w = lane < NT / 32 ? scratch[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int n = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += n;
        }
        if (lane < NT / 32) scratch[lane] = w;
    }
    __syncthreads();
    int add = warp > 0 ? scratch[warp - 1] : 0;
    int total = scratch[NT / 32 - 1];
    __syncthreads();
    scratch[NT / 32] = total;
    return v + add;
}

// Computes W (total units) and the number P = participating_ctas(grid, W, S) of CTAs that take
// part, and positions a cursor at the sequence holding unit u0 of this CTA
// (and, if tail != nullptr, one at the sequence holding its last unit u1 - 1).
// All NT threads must call it.  CTA 0 reports invalid lengths.  Returns false
// when the CTA has no work.
// Block-wide inclusive scan of two ints per thread (one pass for both).
template <int NT>
__device__ __forceinline__ int2 block_scan2_incl(int2 v, int2* scratch /* NT/32 + 1 */) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int nx = __shfl_up_sync(0xffffffffu, v.x, o), ny = __shfl_up_sync(0xffffffffu, v.y, o);
        if (lane >= o) {
            v.x += nx;
            v.y += ny;
        }
    }
    if (lane == 31) scratch[warp] = v;
    __syncthreads();
    int2 add = make_int2(0, 0), tot = make_int2(0, 0);
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) {
        const int2 x = scratch[w];
        if (w < warp) {
            add.x += x.x;
            add.y += x.y;
        }
        tot.x += x.x;
        tot.y += x.y;
    }
    scratch[NT / 32] = tot;      // every thread writes the same value
    return make_int2(v.x + add.x, v.y + add.y);
}

// With seqtab != nullptr and num_seqs <= NT, seqtab[b] receives (L, Q, units
// before b, first q row of b) for every sequence, so that cursors can move on
// without reading global memory (cursor_next with the table).
// With pre_lq != nullptr and num_seqs <= NT, *pre_lq holds this thread's
// (context_lens[tid], q_lens[tid]), already loaded by the caller.
// With bnd != nullptr, num_seqs <= NT and P <= bnd_max, the CTA ranges are cut
// by weight instead (every non-empty segment weighs its units plus ce) into
// the table bnd[0..P] (*bnd_used is set to whether it was), using tmp (int4
// per sequence, scratch for the call) for the sequences' weight prefixes.  A
// range may come out empty only at a segment boundary, and such a CTA has no
// work.
template <int NT, bool CASC = false>
__device__ bool plan_locate(const AttnParams& p, int cta, int ncta, int* scratch, Cursor* cur,
                            int* u0_out, int* u1_out, int* W_out, int* P_out, Cursor* tail = nullptr,
                            int4* seqtab = nullptr, int* bnd = nullptr, int bnd_max = 0, int ce = 0,
                            bool* bnd_used = nullptr, int4* tmp = nullptr, const int2* pre_lq = nullptr) {
    if (bnd_used) *bnd_used = false;
    const int tid = threadIdx.x;
    if (p.num_seqs <= NT) {
        // one chunk: a single load of the lengths and a single two-value scan
        __shared__ int2 s2[NT / 32 + 1];
        __shared__ Cursor s_cur1, s_tail1;
        const int b = tid;
        int L = 0, Q = 0, pb = 0, u = 0, q = 0;
        if (b < p.num_seqs) {
            if (pre_lq) {
                L = pre_lq->x;
                Q = pre_lq->y;
            } else {
                const SeqInfo si = seq_info<CASC>(p, b);
                L = si.L;
                Q = si.Q;
                pb = si.pb;
            }
            if (cta == 0 && seq_error<CASC>(p, L, Q, pb)) raise_error(p.err, PKV_DEVERR_LENGTH);
            u = seq_units<CASC>(p, L, Q, pb);
            q = seq_qrows(Q);
        }
        const int2 inc = block_scan2_incl<NT>(make_int2(u, q), s2);
        if (seqtab && b < p.num_seqs) seqtab[b] = make_int4(L, Q | (pb << 8), inc.x - u, inc.y - q);
        const int W = s2[NT / 32].x;
        const int nseg = p.num_kv_heads / p.hg;                             // segments of a sequence
        const int S = __syncthreads_count(u > 0) * nseg;                   // non-empty segments
        const int P = participating_ctas(ncta, W, S);
        *W_out = W;
        *P_out = P;
        if (cta >= P) return false;
        const int Ub = inc.x - u;
        int u0, u1;
        if (bnd != nullptr && P <= bnd_max) {
            // weighted cut: boundary i sits at weight x = floor(i Wt / P), in the
            // sequence whose weight range holds it; a weight inside a segment's
            // extra ce maps to the segment's end.  One thread per boundary.
            const int w = u + (u > 0 ? ce * nseg : 0);
            const int wincl = block_scan_incl<NT>(w, scratch);
            const int Wt = scratch[NT / 32];
            if (b < p.num_seqs) tmp[b] = make_int4(wincl, Ub, u, 0);
            __syncthreads();
            for (int i = tid; i <= P; i += NT) {
                int v = W;
                if (i < P) {
                    const int x = floor_div_small((long long)i * Wt, P);
                    int lo = 0, hi = p.num_seqs - 1;          // the first sequence with wincl > x
                    while (lo < hi) {
                        const int mid = (lo + hi) >> 1;
                        if (tmp[mid].x > x) hi = mid;
                        else lo = mid + 1;
                    }
                    const int4 e = tmp[lo];                    // (wincl, Ub, units): non-empty
                    const int seglen = e.z / nseg, segw = seglen + ce;
                    const int off = x - (e.x - e.z - ce * nseg);
                    const int j = off / segw, o = off - j * segw;
                    v = e.y + j * seglen + min(o, seglen);
                }
                bnd[i] = v;
            }
            __syncthreads();
            u0 = bnd[cta];
            u1 = bnd[cta + 1];
            if (bnd_used) *bnd_used = true;
        } else {
            u0 = cta_start(cta, W, P);
            u1 = cta_start(cta + 1, W, P);
        }
        *u0_out = u0;
        *u1_out = u1;
        if (u0 >= u1) return false;
        if (b < p.num_seqs && u > 0) {
            Cursor c;
            c.b = b;
            c.Ub = Ub;
            c.qoff = inc.y - q;
            c.L = L;
            c.Q = Q;
            c.pb = pb;
            c.nb = (L + kBlock - 1) / kBlock - pb;
            if (Ub <= u0 && u0 < Ub + u) s_cur1 = c;
            if (Ub <= u1 - 1 && u1 - 1 < Ub + u) s_tail1 = c;
        }
        __syncthreads();
        *cur = s_cur1;
        if (tail) *tail = s_tail1;
        return true;
    }
    const bool one_chunk = p.num_seqs <= NT;      // lengths stay in registers between the passes
    int Lc = 0, Qc = 0, Pc = 0;
    // pass 1: total units
    int total = 0, nonempty = 0;
    for (int base = 0; base < p.num_seqs; base += NT) {
        int b = base + tid;
        int u = 0;
        if (b < p.num_seqs) {
            const SeqInfo si = seq_info<CASC>(p, b);
            if (cta == 0 && seq_error<CASC>(p, si.L, si.Q, si.pb)) raise_error(p.err, PKV_DEVERR_LENGTH);
            u = seq_units<CASC>(p, si.L, si.Q, si.pb);
            Lc = si.L;
            Qc = si.Q;
            Pc = si.pb;
        }
        block_scan_incl<NT>(u, scratch);
        total += scratch[NT / 32];
        nonempty += __syncthreads_count(u > 0);
    }
    const int W = total;
    // With few units, only the first P CTAs take part
    const int P = participating_ctas(ncta, W, nonempty * (p.num_kv_heads / p.hg));
    *W_out = W;
    *P_out = P;
    if (cta >= P) return false;
    const int u0 = cta_start(cta, W, P);
    const int u1 = cta_start(cta + 1, W, P);
    *u0_out = u0;
    *u1_out = u1;
    // pass 2: find b with Ub <= u0 < Ub + units(b) (and the one holding u1 - 1), with q offsets
    __shared__ Cursor s_cur, s_tail;
    int run_u = 0, run_q = 0;
    for (int base = 0; base < p.num_seqs; base += NT) {
        int b = base + tid;
        int u = 0, q = 0, L = 0, Q = 0, pb = 0;
        if (b < p.num_seqs) {
            if (one_chunk) {
                L = Lc;
                Q = Qc;
                pb = Pc;
            } else {
                const SeqInfo si = seq_info<CASC>(p, b);
                L = si.L;
                Q = si.Q;
                pb = si.pb;
            }
            u = seq_units<CASC>(p, L, Q, pb);
            q = seq_qrows(Q);
        }
        int iu = block_scan_incl<NT>(u, scratch);
        int tot_u = scratch[NT / 32];
        __syncthreads();
        int iq = block_scan_incl<NT>(q, scratch);
        int tot_q = scratch[NT / 32];
        __syncthreads();
        int Ub = run_u + iu - u;
        if (b < p.num_seqs && u > 0) {
            Cursor c;
            c.b = b;
            c.Ub = Ub;
            c.qoff = run_q + iq - q;
            c.L = L;
            c.Q = Q;
            c.pb = pb;
            c.nb = (L + kBlock - 1) / kBlock - pb;
            if (Ub <= u0 && u0 < Ub + u) s_cur = c;
            if (Ub <= u1 - 1 && u1 - 1 < Ub + u) s_tail = c;
        }
        run_u += tot_u;
        run_q += tot_q;
    }
    __syncthreads();
    *cur = s_cur;
    if (tail) *tail = s_tail;
    return true;
}

// Advance the cursor to the next sequence with work (all threads, same
// values).  tab: the per-sequence table of plan_locate, or nullptr to read the
// lengths from global memory.
template <bool CASC = false>
__device__ __forceinline__ void cursor_next(const AttnParams& p, Cursor& c, const int4* tab = nullptr) {
    c.Ub += c.nb * p.num_kv_heads;
    c.qoff += seq_qrows(c.Q);
    for (;;) {
        c.b += 1;
        if (c.b >= p.num_seqs) return;
        if (tab) {
            const int4 e = tab[c.b];
            c.L = e.x;
            c.Q = CASC ? (e.y & 0xff) : e.y;
            c.pb = CASC ? (e.y >> 8) : 0;
        } else {
            const SeqInfo si = seq_info<CASC>(p, c.b);
            c.L = si.L;
            c.Q = si.Q;
            c.pb = si.pb;
        }
        if (seq_units<CASC>(p, c.L, c.Q, c.pb) > 0) {
            c.nb = (c.L + kBlock - 1) / kBlock - c.pb;
            return;
        }
        c.qoff += seq_qrows(c.Q);       // skipped sequence: its rows stay packed in q / out
    }
}


// Partial slot of a piece: 0 if its segment started before this CTA's range,
// else 1 (the segment starts here and continues in the next CTA).
__device__ __forceinline__ float* slot_ptr(const AttnParams& p, int cta, int seg_start, int u0) {
    int k = seg_start < u0 ? 0 : 1;
    return p.partials + ((size_t)cta * 2 + k) * (size_t)p.slot_floats;
}

// Merge the partials of segment [S0, S1) (all rows of (b, g)) into out.
// Called by every thread of the CTA that drew the last ticket.
template <int NT>
__device__ void merge_segment(const AttnParams& p, const Cursor& c, int g, int S0, int S1, int W,
                              int ncta, int D) {
    const int c_first = owner_cta(S0, W, ncta), c_last = owner_cta(S1 - 1, W, ncta);
    const int R = p.group * c.Q;
    for (int idx = threadIdx.x; idx < R * D; idx += NT) {
        const int r = idx / D, d = idx % D;
        float M = -INFINITY;
        for (int cc = c_first; cc <= c_last; ++cc) {
            const int u0c = cta_start(cc, W, ncta);
            const float* s = slot_ptr(p, cc, S0, u0c);
            M = fmaxf(M, __ldcg(s + r));
        }
        float den = 0.f, num = 0.f;
        for (int cc = c_first; cc <= c_last; ++cc) {
            const int u0c = cta_start(cc, W, ncta);
            const float* s = slot_ptr(p, cc, S0, u0c);
            const float m = __ldcg(s + r);
            const float w = (m == -INFINITY) ? 0.f : exp2f(m - M);
            den += w * __ldcg(s + p.rows_pad + r);
            num += w * __ldcg(s + 2 * p.rows_pad + (size_t)r * D + d);
        }
        const int i = r / p.group, hl = r % p.group;
        const size_t o = ((size_t)(c.qoff + i) * p.num_q_heads + g * p.group + hl) * D + d;
        p.out[o] = __float2bfloat16_rn(num / den);
    }
}

}  // namespace pkv
