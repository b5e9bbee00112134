// matvec.cu -- the decode matvec (one token): y[o] = row o of the block-quantized
// W against one Q8_0 / Q8_K activation row, for Q4_0, Q8_0, Q4_K, Q6_K and Q2_K,
// and Q4_1, Q5_0, Q5_1, Q5_K.
//
// Design (GB300): the kernel is HBM-bound, so it is built around keeping the
// weight stream in flight.  Each CTA owns a contiguous range of rows (an even
// split of N over the grid).  One thread streams that range into a ring of
// shared-memory stages with 1-D bulk copies (cp.async.bulk, completing on an
// mbarrier) tagged evict-first in L2; the copies cover the 16-byte aligned
// superset of each stage's rows, so no block layout (18, 34, 84, 210 B) needs
// to be aligned.  Meanwhile the CTA unpacks the activation row once into
// shared memory (contiguous int8 codes plus f32 scales and int32 group sums).
// Each row of a stage is then owned by `lpr` lanes of one warp, which decode
// whole blocks from shared memory, take the exact integer block dot with
// __dp4a, fold it into fp32 once per block, and reduce with warp shuffles in a
// fixed order -- so every y[o] is written by one lane, identically on every
// run ([minfer] s3.3: row ownership, no split reduction).
//
// Formulas: [minfer] "10 . CPU matmul: quantized weights x Q8_0 activations"
// s3.2 (the scalar kernels, the K-quant dot walked); [ggml] "ggml Q4_0 vec_dot
// Walkthrough" s1.2 and s2.
#include <stdio.h>

#include "qmm_device.cuh"
#include "qmm_host.h"

namespace qmm {

static __device__ unsigned int g_matvec_error = 0;

constexpr int kThreads = 256;  // blocksums kernel

constexpr int kMaxWarps = 16;  // matvec CTA: up to 16 warps, each with its own ring
constexpr int kMaxGroup = 8;   // weight matrices sharing one activation row in one launch
constexpr int kMaxDepth = 8;   // bulk-copy slots per warp
constexpr uint64_t kSmallCtaBytes = 24 * 1024;  // weight bytes per CTA under which two CTAs share an SM

// The matrices of one launch (all of one format and K): CTAs
// [cta_end[g-1], cta_end[g]) own matrix g and split its N[g] rows evenly.
struct MatSet {
    const uint8_t* W[kMaxGroup];
    float* y[kMaxGroup];
    int N[kMaxGroup];
    int cta_end[kMaxGroup];
    int G;
    const float* gamma;  // fused quantize: RMSNorm the row first with this weight (null: no norm)
    float eps;
    uint32_t norm_off;   // shared-memory offset of the norm's K/8 partial sums
};

struct MatvecPlan {
    bool su;              // decode whole super-units (Q8_0 / Q4_0 with K % 256 == 0)
    int nw;               // warps per CTA
    int lpr;              // lanes per row (power of two, 1..32)
    int pieces;           // segments per row
    int piece_units;      // units per segment (the last segment of a row may have fewer)
    int item_segs;        // segments per item (whole passes of 32 / lpr segments)
    uint32_t part_off;    // shared offset of the per-segment partial sums (pieces > 1)
    int depth;            // slots in each warp's ring
    uint32_t slot_bytes;  // bytes per slot (the item's 16-byte aligned superset)
    uint32_t act_bytes;   // shared bytes before the first slot (barriers, activation)
    uint32_t smem;        // total dynamic shared memory
    uint32_t norm_off;    // a normed row's partial sums
    int grid;
};

__host__ __device__ inline uint32_t align_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

// activation region: [codes][scales: 4*nd B][sums], 128-byte padded; Q8_0:
// K code bytes and nd int32 sums; Q8_K: 16 chunk rows of pitch q8k_pitch(nd)
// and 8 bsum-pair rows of the same pitch
__host__ __device__ inline uint32_t act_code_bytes(int act, int K) {
    return act == QMM_Q8_0 ? (uint32_t)K : 256u * (uint32_t)q8k_pitch(K / 256);
}
__host__ __device__ inline uint32_t act_region_bytes(int act, int K) {
    const int nd = act == QMM_Q8_0 ? K / 32 : K / 256;
    const uint32_t sum_bytes = act == QMM_Q8_0 ? 4u * nd : 32u * (uint32_t)q8k_pitch(nd);
    return align_up(act_code_bytes(act, K) + 4u * nd + sum_bytes, 128u);
}

template <int WT>
__device__ __forceinline__ float unit_contrib(const SmemBytes& w, uint32_t o, const ActView& a, int u) {
    if constexpr (WT == QMM_Q4_0 || WT == QMM_Q8_0 || WT == QMM_Q5_0) {
        uint32_t db;
        const int isum = (WT == QMM_Q4_0)   ? q4_0_isum(w, o, a, u, &db)
                         : (WT == QMM_Q8_0) ? q8_0_isum(w, o, a, u, &db)
                                            : q5_0_isum(w, o, a, u, &db);
        return (float)isum * h2f(db) * a.d[u];
    } else if constexpr (WT == QMM_Q4_1 || WT == QMM_Q5_1) {
        uint32_t dm;
        const int isum = (WT == QMM_Q4_1) ? q4_1_isum(w, o, a, u, &dm) : q5_1_isum(w, o, a, u, &dm);
        // d*dx*sum(q*a) + m*dx*sum(a): the min meets the activation block's code sum
        return (float)isum * h2f(dm & 0xFFFFu) * a.d[u] + (float)a.s[u] * h2f(dm >> 16) * a.d[u];
    } else if constexpr (WT == QMM_Q6_K) {
        int v, m;
        uint32_t db;
        q6_K_isums(w, o, a, u, &v, &m, &db);
        const float d = h2f(db) * a.d[u];
        return d * (float)(v - 32 * m);
    } else {
        int v, m;
        uint32_t db, dmb;
        if constexpr (WT == QMM_Q4_K) q4_K_isums(w, o, a, u, &v, &m, &db, &dmb);
        else if constexpr (WT == QMM_Q5_K) q5_K_isums(w, o, a, u, &v, &m, &db, &dmb);
        else q2_K_isums(w, o, a, u, &v, &m, &db, &dmb);
        const float d = h2f(db) * a.d[u];
        const float dmin = h2f(dmb) * a.d[u];
        // the page's order: subtract the min term, then add the value term
        return -(dmin * (float)m) + d * (float)v;
    }
}

// Rows cut into `pieces` segments of `piece_units` units (the last may be
// shorter); segment s = row s / pieces, piece s % pieces.  A unit is a block,
// a super-block or a super-unit (ubytes each).  Segments are consecutive in W.
template <bool SPLIT>
struct SegGeom {
    uint64_t rb;      // row bytes
    int nunit;        // units per row
    int pieces;       // 1 unless SPLIT
    int piece_units;
    int ubytes;
    __device__ __forceinline__ uint64_t off(int s) const {  // byte offset of segment s in W
        if constexpr (!SPLIT) return (uint64_t)s * rb;
        const int row = s / pieces, piece = s - row * pieces;
        const int u = min(piece * piece_units, nunit);
        return (uint64_t)row * rb + (uint64_t)u * ubytes;
    }
};

// Issues the bulk copy of the bytes [g0, g1) of W, as their 16-byte aligned
// superset (the last < 16 bytes of W excepted), into a slot.
__device__ __forceinline__ void issue_item(const uint8_t* W, uint64_t g0, uint64_t g1, uint64_t total_al,
                                           uint8_t* slot, uint32_t bar, uint64_t pol, uint32_t slot_bytes) {
    const uint64_t a0 = g0 & ~15ull;
    uint64_t a1 = (g1 + 15ull) & ~15ull;
    if (a1 > total_al) a1 = total_al;
    uint32_t bytes = a1 > a0 ? (uint32_t)(a1 - a0) : 0u;
    if (!QMM_IN_BOUNDS(g_matvec_error, bytes, (int64_t)slot_bytes + 1)) bytes = 0;  // the copy must fit its slot
    mbar_arrive_expect_tx(bar, bytes);
    if (bytes) bulk_g2s(smem_u32(slot), W + a0, bytes, bar, pol);
}

// The decode matvec.  Each CTA owns an even share of the rows.  A row is one
// segment, or `pieces` segments when it is long enough that one segment would
// leave lanes idle; the CTA's segments are cut into items of `item_segs`
// consecutive segments (whole passes of 32 / lpr segments).  Warp w of the CTA
// takes items w, w + nw, w + 2nw, ... and streams them through its own ring of
// `depth` shared-memory slots with 1-D bulk copies (cp.async.bulk completing
// on the slot's mbarrier, evict-first in L2).  A warp refills a slot as soon as
// it has decoded it, so no warp waits for another and no CTA-wide barrier sits
// in the stream.  Lanes take the units of a segment (a block, a super-block or,
// with SU, a super-unit of 8 blocks) in steps of `lpr`, decode them from shared
// memory, take the exact integer block dots with dp4a, fold each into fp32 once
// per block and reduce with shuffles in a fixed order.  A one-segment row is
// written by that lane; otherwise the segments' partial sums meet in shared
// memory and one thread adds them in piece order.  Either way every y[o] comes
// from one fixed order of operations, identical on every run ([minfer] "10 .
// CPU matmul: quantized weights x Q8_0 activations" s3.3: row ownership).
//
// With pdl set the kernel is one link of a programmatic-dependent-launch chain:
// it lets its successor launch at once and streams the first item of each warp
// (the weights, which nothing writes) before it waits for its predecessor's
// grid; only then does it read the activation, issue the remaining copies and
// write y.  Few copies are in flight while the activation is read, so its
// loads are not queued behind the whole weight stream (Q8_0 weights with
// several items per warp request the rest once the row's loads are out).
//
// A Q8_0 activation block (f16 scale bits, 8 code words) into the layout the
// decoder of WT reads.
template <int WT, bool SU>
__device__ __forceinline__ void put_act_block(const uint32_t w[8], uint32_t dbits, int b, int nb, int nsu, uint8_t* aq,
                                              float* ad, int* as) {
    if constexpr (SU && (WT == QMM_Q8_0 || WT == QMM_Q4_0))
        su_put_block<WT == QMM_Q4_0>(w, dbits, b, nsu, aq, ad, as);
    else if constexpr (SU)
        su_put_halves(w, dbits, b, nsu, aq, ad, as);
    else
        act_put_q8_0_block(w, dbits, b, nb, aq, ad, as);
}

// the 34-byte block b of the quantized row (16-bit stores: rows of a larger
// buffer are only 2-byte aligned)
__device__ __forceinline__ void store_q8_0_block(uint8_t* xq_out, int b, uint32_t dbits, const uint32_t w[8]) {
    unsigned short* o = reinterpret_cast<unsigned short*>(xq_out + (size_t)b * 34);
    o[0] = (unsigned short)dbits;
#pragma unroll
    for (int i = 0; i < 8; i++) {
        o[1 + 2 * i] = (unsigned short)(w[i] & 0xFFFFu);
        o[2 + 2 * i] = (unsigned short)(w[i] >> 16);
    }
}

// The fused quantize of the whole row in one pass, LPB lanes per block (the
// caller has checked K/32 * LPB <= threads).  FUSE 2 norms each value first.
// after_loads() runs once the row's loads are issued, before their values are used.
template <int WT, bool SU, int FUSE, int LPB, class AfterLoads>
__device__ __forceinline__ void fused_q8_0_lanes(const float* x, const float* gamma, float sn, uint8_t* xq_out, int K,
                                                 int nsu, uint8_t* aq, float* ad, int* as, AfterLoads&& after_loads) {
    constexpr int NV = 8 / LPB;
    const int nb = K / 32, tid = threadIdx.x;
    const int b = tid / LPB, part = tid - b * LPB;
    const bool active = b < nb;
    const size_t off = (size_t)(active ? b : 0) * 8 + (size_t)part * NV;
    float4 v[NV];
#pragma unroll
    for (int i = 0; i < NV; i++) v[i] = active ? reinterpret_cast<const float4*>(x)[off + i] : make_float4(0.f, 0.f, 0.f, 0.f);
    after_loads();
    if constexpr (FUSE == 2) {
#pragma unroll
        for (int i = 0; i < NV; i++)
            if (active) v[i] = norm4(v[i], sn, reinterpret_cast<const float4*>(gamma)[off + i]);
    }
    uint32_t w[8], dbits;
    quant_q8_0_block_lanes<LPB>(v, part, &dbits, w);
    if (active && part == 0) {
        if (blockIdx.x == 0 && xq_out != nullptr) store_q8_0_block(xq_out, b, dbits, w);
        put_act_block<WT, SU>(w, dbits, b, nb, nsu, aq, ad, as);
    }
}

// With FUSE (1) the kernel takes the f32 activation row x instead of xq and
// quantizes it itself (every CTA, into shared memory, with the same per-block
// arithmetic as the standalone quantizer, so the codes are the same bytes);
// CTA 0 also stores the quantized row to xq_out when that is not null.  One
// launch then does the whole quantize + multiply of a decode token.  FUSE 2
// RMSNorms the row first (set.gamma, set.eps); a mode of its own, so the plain
// fused kernel carries none of it.
template <int WT, bool SU, int FUSE, bool SPLIT>
__global__ void __launch_bounds__(kMaxWarps * 32, 1) matvec_kernel(const __grid_constant__ MatSet set,
                                                                  const uint8_t* __restrict__ xq,
                                                                  const float* __restrict__ x, uint8_t* xq_out,
                                                                  int K, int lpr,
                                                                  int pieces, int piece_units, int item_segs,
                                                                  int depth, uint32_t slot_bytes, uint32_t part_off,
                                                                  uint32_t act_bytes, int pdl) {
    using F = Fmt<WT>;
    if (pdl) pdl_launch_dependents();
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nw = blockDim.x >> 5;
    // this CTA's matrix, and its place among the CTAs of that matrix
    int g = 0;
    while (g + 1 < set.G && (int)blockIdx.x >= set.cta_end[g]) g++;
    const int cta0 = g ? set.cta_end[g - 1] : 0;
    const int ncta = set.cta_end[g] - cta0, bl = (int)blockIdx.x - cta0;
    const uint8_t* __restrict__ W = set.W[g];
    float* __restrict__ y = set.y[g];
    const int N = set.N[g];
    // [barriers: nw * depth][activation][slots: nw * depth * slot_bytes]
    uint64_t* full = reinterpret_cast<uint64_t*>(smem) + warp * depth;
    uint8_t* aq = smem + align_up(8u * nw * depth, 128u);
    const int nd = F::ACT == QMM_Q8_0 ? K / 32 : K / 256;
    const int nsu = K / 256;
    const int ap = F::ACT == QMM_Q8_0 ? nd : q8k_pitch(nd);  // the view's pitch
    const int qbytes = SU ? SuFmt<has_su<WT>() ? WT : QMM_Q8_0>::A * nsu : (int)act_code_bytes(F::ACT, K);
    float* ad = reinterpret_cast<float*>(aq + qbytes);
    int* as = reinterpret_cast<int*>(ad + nd);
    uint8_t* slots = smem + act_bytes + (size_t)warp * depth * slot_bytes;

    const int units = K / F::BV;
    const uint64_t rb = (uint64_t)units * F::BB;
    if constexpr (!SPLIT) pieces = 1;
    const SegGeom<SPLIT> geo{rb, SU ? nsu : units, pieces, piece_units,
                             SU ? SuFmt<has_su<WT>() ? WT : QMM_Q8_0>::W : F::BB};
    // an even split of the matrix's rows: its first N % ncta CTAs take one row more
    const int rq = N / ncta, rr = N - rq * ncta;
    const int r_begin = bl * rq + min(bl, rr);
    const int r_end = r_begin + rq + (bl < rr ? 1 : 0);
    const int s_begin = r_begin * pieces, s_end = r_end * pieces;  // this CTA's segments
    const int nitems = (s_end - s_begin + item_segs - 1) / item_segs;
    const int my_items = nitems > warp ? (nitems - warp + nw - 1) / nw : 0;
    const uint64_t total = (uint64_t)N * rb;
    const uint64_t total_al = total & ~15ull;

    uint64_t pol = 0;
    if (lane == 0) {
        for (int i = 0; i < depth; i++) mbar_init(smem_u32(&full[i]), 1);
        fence_mbar_init();
        pol = policy_evict_first();
        if (my_items > 0) {
            const int s0 = s_begin + warp * item_segs;
            issue_item(W, geo.off(s0), geo.off(min(s0 + item_segs, s_end)), total_al, slots, smem_u32(&full[0]), pol,
                       slot_bytes);
        }
    }
    __syncwarp();

    // the rest of this warp's ring (its first slot was requested above)
    auto issue_rest = [&] {
        for (int k = 1; k < depth && k < my_items; k++) {
            const int s0 = s_begin + (warp + k * nw) * item_segs;
            issue_item(W, geo.off(s0), geo.off(min(s0 + item_segs, s_end)), total_al, slots + (size_t)k * slot_bytes,
                       smem_u32(&full[k]), pol, slot_bytes);
        }
    };
    bool early = false;  // issue_rest ran right after the activation's loads

    if (pdl) pdl_wait();  // the activation row comes from the previous kernel
    {
        const int nthr = blockDim.x;
        float sn = 1.0f;  // the RMSNorm scale of the row, when the fused quantize norms it first
        if constexpr (FUSE == 2) sn = rms_scale(x, K, reinterpret_cast<float*>(smem + set.norm_off), set.eps);
        if constexpr (F::ACT == QMM_Q8_0) {
            // one thread per activation block: read (or, with FUSE, quantize)
            // its 32 codes and put them in the layout the decoder reads; a
            // fused quantize that fits in one pass takes 4 or 2 lanes per block
            const int nb = K / 32;
            int lpb = 1;
            if constexpr (FUSE) lpb = nb * 4 <= nthr ? 4 : (nb * 2 <= nthr ? 2 : 1);
            if constexpr (FUSE) {
                // Q8_0 weights with at least two items per warp request the rest of each
                // ring as soon as the row's loads are out, not after the row is in place
                // (12288 x 4096 step 9.56 -> 9.20 us); for the other formats, and for
                // smaller Q8_0 matrices, the earlier requests measured slower.
                early = WT == QMM_Q8_0 && nitems >= 2 * nw && lpb > 1;
                auto rest = [&] {
                    if (early && lane == 0) issue_rest();
                };
                if (lpb == 4) fused_q8_0_lanes<WT, SU, FUSE, 4>(x, set.gamma, sn, xq_out, K, nsu, aq, ad, as, rest);
                if (lpb == 2) fused_q8_0_lanes<WT, SU, FUSE, 2>(x, set.gamma, sn, xq_out, K, nsu, aq, ad, as, rest);
            }
            // the same early request on a quantized Q8_0 row (unsplit rows only: the split
            // 4096 x 12288 matrix measured 0.1 us slower; 12288 x 4096: 9.09 -> 8.92 us)
            const bool early0 = !FUSE && !SPLIT && WT == QMM_Q8_0 && nitems >= 2 * nw;
            bool done0 = false;
            for (int b = tid; lpb == 1 && b < nb; b += nthr) {
                uint32_t w[8], dbits;
                if constexpr (FUSE) {
                    const float4* x4 = reinterpret_cast<const float4*>(x) + (size_t)b * 8;
                    float4 v[8];
#pragma unroll
                    for (int i = 0; i < 8; i++) v[i] = x4[i];
                    if constexpr (FUSE == 2) {
                        const float4* g4 = reinterpret_cast<const float4*>(set.gamma) + (size_t)b * 8;
#pragma unroll
                        for (int i = 0; i < 8; i++) v[i] = norm4(v[i], sn, g4[i]);
                    }
                    quant_q8_0_block(v, &dbits, w);
                    if (blockIdx.x == 0 && xq_out != nullptr) store_q8_0_block(xq_out, b, dbits, w);
                } else {
                    const unsigned short* p = reinterpret_cast<const unsigned short*>(xq + (size_t)b * 34);
                    dbits = p[0];
#pragma unroll
                    for (int i = 0; i < 8; i++) w[i] = (uint32_t)p[1 + 2 * i] | ((uint32_t)p[2 + 2 * i] << 16);
                    if (early0 && !done0 && lane == 0) issue_rest();
                    done0 = true;
                }
                put_act_block<WT, SU>(w, dbits, b, nb, nsu, aq, ad, as);
            }
            if (early0) {  // a warp with no block of the row still requests its ring
                if (!done0 && lane == 0) issue_rest();
                early = true;
            }
        } else {
            if constexpr (FUSE) {
                // one warp per super-block, both rounds of loads issued first
                const float4* x4 = reinterpret_cast<const float4*>(x);
                for (int b0 = warp; b0 < nd; b0 += 2 * nw) {
                    const int b1 = b0 + nw;
                    float4 v0 = x4[b0 * 64 + 2 * lane], v1 = x4[b0 * 64 + 2 * lane + 1];
                    float4 v2 = make_float4(0.f, 0.f, 0.f, 0.f), v3 = v2;
                    if (b1 < nd) v2 = x4[b1 * 64 + 2 * lane], v3 = x4[b1 * 64 + 2 * lane + 1];
                    if constexpr (FUSE == 2) {
                        const float4* g4 = reinterpret_cast<const float4*>(set.gamma);
                        v0 = norm4(v0, sn, g4[b0 * 64 + 2 * lane]);
                        v1 = norm4(v1, sn, g4[b0 * 64 + 2 * lane + 1]);
                        if (b1 < nd) {
                            v2 = norm4(v2, sn, g4[b1 * 64 + 2 * lane]);
                            v3 = norm4(v3, sn, g4[b1 * 64 + 2 * lane + 1]);
                        }
                    }
                    // straight into the decoder's layout; CTA 0 also stores the row
                    uint8_t* ob = blockIdx.x == 0 ? xq_out : nullptr;
                    quant_q8_K_lane_put(v0, v1, lane, b0, ap, aq, ad, as, ob ? ob + b0 * 292 : nullptr);
                    if (b1 < nd) quant_q8_K_lane_put(v2, v3, lane, b1, ap, aq, ad, as, ob ? ob + b1 * 292 : nullptr);
                }
            } else {
                unpack_q8_K_row_by(xq, nd, ap, aq, ad, as, tid, nthr);
            }
        }
        __syncthreads();
    }
    if (lane == 0 && !early) issue_rest();

    const ActView act{aq, ad, as, ap};
    float* part = reinterpret_cast<float*>(smem + part_off);  // pieces > 1: one partial per segment
    const int segs_per_pass = 32 / lpr;
    const int ssub = lane / lpr, li = lane % lpr;
    bool failed = false;
    for (int k = 0; k < my_items; k++) {
        const int slot = k % depth;
        const bool ok = mbar_wait_bounded(smem_u32(&full[slot]), (uint32_t)(k / depth) & 1u, kWaitLimitNs);
        if (__any_sync(0xffffffffu, !ok)) {
            if (lane == 0) atomicOr(&g_matvec_error, kErrTimeout);
            failed = true;
            break;
        }
        const int s0 = s_begin + (warp + k * nw) * item_segs;
        const int s1 = min(s0 + item_segs, s_end);
        const uint64_t a0 = geo.off(s0) & ~15ull;
        uint8_t* sbuf = slots + (size_t)slot * slot_bytes;
        const SmemBytes wv{sbuf};
        for (int ss = s0; ss < s1; ss += segs_per_pass) {
            const int seg = ss + ssub;
            if (seg == (SPLIT ? N * pieces : N) - 1 && total > total_al) {
                // the last < 16 bytes of W lie in the last segment: not reachable
                // by a 16-byte bulk copy, so this warp fetches them itself
                for (uint64_t i = total_al + li; i < total; i += lpr)
                    if (QMM_IN_BOUNDS(g_matvec_error, i - a0, slot_bytes)) sbuf[i - a0] = W[i];
            }
            __syncwarp();
            float acc = 0.0f;
            if (seg < s1) {
                int u0 = 0, un = geo.nunit;
                if constexpr (SPLIT) {
                    const int piece = seg - (seg / pieces) * pieces;
                    u0 = piece * piece_units;
                    un = min(piece_units, geo.nunit - u0);
                }
                const uint32_t so = (uint32_t)(geo.off(seg) - a0);
                // the segment's bytes must lie inside the slot the item was copied to
                const int64_t seg_end = (int64_t)so + (int64_t)un * (SU ? geo.ubytes : F::BB);
                if (!QMM_IN_BOUNDS(g_matvec_error, seg_end - 1, slot_bytes)) un = 0;
                if constexpr (SU) {
                    for (int u = li; u < un; u += lpr) {
                        const int ug = u0 + u;
                        if constexpr (WT == QMM_Q8_0) acc += su_q8_0(sbuf + so + 272u * u, aq, nsu, ug, ad + 8 * ug);
                        else if constexpr (WT == QMM_Q4_0)
                            acc += su_q4_0(sbuf + so + 144u * u, aq, nsu, ug, ad + 8 * ug, as + 8 * ug);
                        else if constexpr (has_su<WT>())
                            acc += su_q45<WT>(sbuf + so + (uint32_t)SuFmt<WT>::W * u, aq, nsu, ug, ad + 8 * ug,
                                              as + 8 * ug);
                    }
                } else {
#pragma unroll 4
                    for (int u = li; u < un; u += lpr)
                        acc += unit_contrib<WT>(wv, so + (uint32_t)(u * F::BB), act, u0 + u);
                }
            }
            for (int off = lpr >> 1; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            if (seg < s1 && li == 0) {
                if constexpr (SPLIT) {
                    if (QMM_IN_BOUNDS(g_matvec_error, seg - s_begin, s_end - s_begin)) part[seg - s_begin] = acc;
                } else if (QMM_IN_BOUNDS(g_matvec_error, seg, N)) {
                    y[seg] = acc;
                }
            }
        }
        __syncwarp();
        if (lane == 0 && k + depth < my_items) {
            const int q0 = s_begin + (warp + (k + depth) * nw) * item_segs;
            issue_item(W, geo.off(q0), geo.off(min(q0 + item_segs, s_end)), total_al, sbuf, smem_u32(&full[slot]),
                       pol, slot_bytes);
        }
    }
    if constexpr (SPLIT) {
        // a row's pieces were taken by different warps: add them in piece order
        if (!__syncthreads_or(failed ? 1 : 0)) {
            for (int r = r_begin + tid; r < r_end; r += blockDim.x) {
                float v = 0.0f;
                for (int p = 0; p < pieces; p++) v += part[(r - r_begin) * pieces + p];
                if (QMM_IN_BOUNDS(g_matvec_error, r, N)) y[r] = v;
            }
        }
    }
}

// ------------------------------------------------------------------ blocksums (verification)
// One CTA per (token, group of rows): copies the rows' bytes into shared memory
// with plain loads and runs the same decoders, writing the integers.
template <int WT>
__global__ void __launch_bounds__(kThreads) blocksums_kernel(const uint8_t* __restrict__ W,
                                                             const uint8_t* __restrict__ xq, int32_t* __restrict__ out,
                                                             int N, int K, int rows_per_cta, uint32_t act_bytes) {
    using F = Fmt<WT>;
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* aq = smem + 128;
    const int nd = F::ACT == QMM_Q8_0 ? K / 32 : K / 256;
    const int ap = F::ACT == QMM_Q8_0 ? nd : q8k_pitch(nd);
    float* ad = reinterpret_cast<float*>(aq + act_code_bytes(F::ACT, K));
    int* as = reinterpret_cast<int*>(ad + nd);
    uint8_t* wbuf = smem + act_bytes;

    const int t = blockIdx.y;
    const int units = K / F::BV;
    const uint64_t rb = (uint64_t)units * F::BB;
    const uint64_t xrb = F::ACT == QMM_Q8_0 ? (uint64_t)(K / 32) * Q8_0_BB : (uint64_t)(K / 256) * Q8_K_BB;
    const uint8_t* xrow = xq + (uint64_t)t * xrb;
    if constexpr (F::ACT == QMM_Q8_0) unpack_q8_0_row(xrow, K, aq, ad, as);
    else unpack_q8_K_row(xrow, K, aq, ad, as);

    const int r0 = blockIdx.x * rows_per_cta;
    const int r1 = min(r0 + rows_per_cta, N);
    const uint64_t a0 = ((uint64_t)r0 * rb) & ~15ull;
    const uint64_t g1 = (uint64_t)r1 * rb;
    for (uint64_t i = a0 + threadIdx.x; i < g1; i += blockDim.x)
        if (QMM_IN_BOUNDS(g_matvec_error, i - a0, (uint64_t)rows_per_cta * rb + 16)) wbuf[i - a0] = W[i];
    __syncthreads();

    const ActView act{aq, ad, as, ap};
    const SmemBytes wv{wbuf};
    const int per = F::ACT == QMM_Q8_0 ? units : 2 * units;
    for (int i = threadIdx.x; i < (r1 - r0) * units; i += blockDim.x) {
        const int row = r0 + i / units, u = i % units;
        const uint32_t o = (uint32_t)((uint64_t)row * rb - a0) + (uint32_t)(u * F::BB);
        int32_t* dst = out + ((uint64_t)t * N + row) * per;
        if (!QMM_IN_BOUNDS(g_matvec_error, ((uint64_t)t * N + row) * per + u * (per / units), (uint64_t)gridDim.y * N * per))
            continue;
        uint32_t db, dmb;
        int v = 0, m = 0;
        if constexpr (WT == QMM_Q4_0) v = q4_0_isum(wv, o, act, u, &db);
        else if constexpr (WT == QMM_Q8_0) v = q8_0_isum(wv, o, act, u, &db);
        else if constexpr (WT == QMM_Q4_K) q4_K_isums(wv, o, act, u, &v, &m, &db, &dmb);
        else if constexpr (WT == QMM_Q2_K) q2_K_isums(wv, o, act, u, &v, &m, &db, &dmb);
        else if constexpr (WT == QMM_Q6_K) q6_K_isums(wv, o, act, u, &v, &m, &db);
        else if constexpr (WT == QMM_Q4_1) v = q4_1_isum(wv, o, act, u, &db);
        else if constexpr (WT == QMM_Q5_0) v = q5_0_isum(wv, o, act, u, &db);
        else if constexpr (WT == QMM_Q5_1) v = q5_1_isum(wv, o, act, u, &db);
        else q5_K_isums(wv, o, act, u, &v, &m, &db, &dmb);
        if constexpr (F::ACT == QMM_Q8_0) {
            dst[u] = v;
        } else {
            dst[2 * u] = v;
            dst[2 * u + 1] = m;
        }
    }
}

// ------------------------------------------------------------------ host side
qmm_status current_device(DeviceInfo* info) {
    static DeviceInfo cache[64];
    static PerDeviceOnce once;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return QMM_E_CUDA;
    const qmm_status st = once.run(dev, [&] {
        DeviceInfo d;
        d.device = dev;
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return QMM_E_CUDA;
        if (cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
            return QMM_E_CUDA;
        if (cudaDeviceGetAttribute(&d.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess)
            return QMM_E_CUDA;
        if (cudaDeviceGetAttribute(&d.smem_reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess)
            return QMM_E_CUDA;
        cache[dev] = d;
        return QMM_OK;
    });
    if (st != QMM_OK) return st;
    *info = cache[dev];
    return QMM_OK;
}

// activation bytes in shared memory for a plan (without the barriers)
__host__ inline uint32_t matvec_act_bytes(int wt, int act, int K, bool su) {
    if (!su) return act_region_bytes(act, K);
    const int nsu = K / 256, nd = K / 32;
    const int per = wt == QMM_Q4_0 ? 288 : (wt == QMM_Q8_0 ? 272 : 256);
    return align_up((uint32_t)(per * nsu + 8 * nd), 128u);
}

// Picks the launch shape for G matrices of one format and K (G = 1: a plain
// matvec).  A row is cut into the fewest segments that keep the most lanes busy
// (a segment of U units gets the smallest power of two >= U lanes; at most 32).
// Lanes per segment cover its units (a pass = 32 / lpr segments); an item is
// one pass, or several when a pass is under 4 KB.  The SMs are shared among the
// matrices in proportion to their rows, one CTA per SM.  Each warp keeps two
// items in flight when 12 or more warps fit that way, else one item with 16
// warps (more warps beat a deeper ring there).
template <int WT>
static qmm_status plan_matvec(const int64_t* Ns, int G, int64_t K, const DeviceInfo& dev, bool fuse, bool norm,
                              MatvecPlan* p, int* cta_end) {
    using F = Fmt<WT>;
    p->su = has_su<WT>() && K % 256 == 0;
    const int nunit = p->su ? (int)(K / 256) : (int)(K / F::BV);
    const int ubytes = p->su ? 8 * F::BB : F::BB;
    int best_p = 1, best_l = 32;
    double best_use = -1.0;
    for (int cap = 32; cap >= 8; cap >>= 1) {
        const int P = (nunit + cap - 1) / cap, U = (nunit + P - 1) / P;
        int l = 1;
        while (l < U) l <<= 1;
        const double use = (double)nunit / ((double)P * l);
        if (use > best_use + 1e-9) best_use = use, best_p = P, best_l = l;
    }
    p->pieces = best_p;
    p->piece_units = (nunit + best_p - 1) / best_p;
    p->lpr = best_l;
    // Q4_0 super-units: two per lane (two independent chains per lane, and a
    // warp's per-pass overhead over twice the bytes) measured 6% faster at
    // 12288 x 4096; the other formats were slower that way
    if (WT == QMM_Q4_0 && p->su && p->lpr >= 16 && p->piece_units >= p->lpr) p->lpr >>= 1;
    // short rows of 32-value blocks (no super-units): 4 lanes per row, several
    // blocks per lane and 8 rows per pass, rather than one row per 32-lane pass
    // of short dependency chains (Q4_0 4864 x 896: 4.02 -> 2.22 us; 8 lanes gave
    // 2.85, 2 lanes 2.35)
    if (!p->su && F::BV == 32 && p->pieces == 1 && nunit >= 8 && nunit <= 32) p->lpr = 4;
    const uint64_t seg_bytes = (uint64_t)p->piece_units * ubytes;
    const int spp = 32 / p->lpr;
    const uint64_t pass_bytes = (uint64_t)spp * seg_bytes;
    int npass = (int)(4096u / pass_bytes);
    if (npass < 1) npass = 1;
    p->item_segs = npass * spp;
    const uint64_t sb = align_up((uint32_t)(npass * pass_bytes + 32), 128u);
    if (sb > 0x7FFFFFFFull) return QMM_E_SHAPE;
    p->slot_bytes = (uint32_t)sb;

    // CTAs per matrix: a share of the SMs proportional to its rows, at least one,
    // at most one per item and per row
    int64_t total_rows = 0, cap[kMaxGroup];
    for (int g = 0; g < G; g++) {
        total_rows += Ns[g];
        cap[g] = (Ns[g] * p->pieces + p->item_segs - 1) / p->item_segs;
        if (cap[g] > Ns[g]) cap[g] = Ns[g];
    }
    int grid[kMaxGroup];
    int64_t sum = 0;
    for (int g = 0; g < G; g++) {
        int64_t c = (int64_t)((double)dev.sms * (double)Ns[g] / (double)total_rows + 0.5);
        if (c < 1) c = 1;
        if (c > cap[g]) c = cap[g];
        grid[g] = (int)c;
        sum += c;
    }
    // trim an overshoot from the largest shares (the SMs run one CTA each)
    while (sum > dev.sms) {
        int gm = -1;
        for (int g = 0; g < G; g++)
            if (grid[g] > 1 && (gm < 0 || grid[g] > grid[gm])) gm = g;
        if (gm < 0) break;
        grid[gm]--;
        sum--;
    }
    uint64_t rows_max = 1;
    int acc = 0;
    for (int g = 0; g < G; g++) {
        acc += grid[g];
        cta_end[g] = acc;
        const uint64_t r = (uint64_t)((Ns[g] + grid[g] - 1) / grid[g]);
        if (r > rows_max) rows_max = r;
    }
    p->grid = acc;

    uint32_t act = matvec_act_bytes(WT, F::ACT, (int)K, p->su);
    // a normed row: the K/8 partial sums of squares after the activation
    const uint32_t norm_rel = act;
    // (sized for any block of up to kMaxWarps warps)
    if (norm) act += align_up(4u * (uint32_t)rms_scratch_bound((int)K, kMaxWarps * 32), 128u);
    const uint64_t part_bytes = p->pieces > 1 ? align_up((uint32_t)(rows_max * p->pieces * 4), 128u) : 0;
    const uint32_t bar_max = align_up(8u * kMaxWarps * kMaxDepth, 128u);
    if ((uint64_t)dev.max_smem_optin < (uint64_t)bar_max + act + part_bytes + sb) return QMM_E_SHAPE;
    // A CTA with little to stream (a small matrix) gets at most 8 warps and half
    // an SM's shared memory: two CTAs then fit on an SM, so the CTAs of the next
    // launch in a chain start while this launch's CTAs are still finishing.
    uint64_t cta_bytes = 0;
    for (int g = 0; g < G; g++) {
        const uint64_t b = (uint64_t)((Ns[g] + grid[g] - 1) / grid[g]) * (uint64_t)(K / F::BV) * F::BB;
        if (b > cta_bytes) cta_bytes = b;
    }
    uint64_t smem_cap = (uint64_t)dev.max_smem_optin;
    int nw_cap = kMaxWarps;
    const uint64_t half_sm = (uint64_t)dev.smem_per_sm / 2 - (uint64_t)dev.smem_reserved;
    if (cta_bytes <= kSmallCtaBytes && half_sm >= (uint64_t)bar_max + act + part_bytes + 2 * sb &&
        half_sm < smem_cap) {
        smem_cap = half_sm;
        nw_cap = kMaxWarps / 2;
    }
    const uint64_t budget = smem_cap - bar_max - act - part_bytes;
    int nw = (int)(budget / (2 * sb));
    if (nw >= 12 || (nw_cap < kMaxWarps && nw >= 1)) {
        p->depth = 2;
    } else {
        p->depth = 1;
        nw = (int)(budget / sb);
    }
    if (nw > nw_cap) nw = nw_cap;
    if (nw < 1) return QMM_E_SHAPE;
    // a deeper ring when the shared memory holds more of a warp's items: with
    // only a few items per warp, a ring of two makes each warp wait for several
    // full memory round trips, where all of its items could be in flight at once
    {
        const uint64_t items_cta = (rows_max * (uint64_t)p->pieces + p->item_segs - 1) / p->item_segs;
        const int ipw = (int)((items_cta + nw - 1) / nw);
        uint64_t dmax = budget / ((uint64_t)nw * sb);
        if (dmax > (uint64_t)kMaxDepth) dmax = kMaxDepth;
        if (ipw > p->depth && (int)dmax > p->depth) p->depth = ipw < (int)dmax ? ipw : (int)dmax;
    }
    p->nw = nw;
    p->part_off = align_up(8u * nw * p->depth, 128u) + act;
    p->norm_off = align_up(8u * nw * p->depth, 128u) + norm_rel;
    p->act_bytes = p->part_off + (uint32_t)part_bytes;
    p->smem = p->act_bytes + (uint32_t)(nw * p->depth) * p->slot_bytes;
    return QMM_OK;
}

template <int WT, bool SU, int FUSE, bool SPLIT>
static qmm_status launch_matvec_k(const MatSet& set, const void* xq, const float* x, void* xq_out, int64_t K,
                                   const MatvecPlan& p, const DeviceInfo& dev, cudaStream_t stream, bool pdl) {
    static PerDeviceOnce attr_once;
    const qmm_status ast = attr_once.run(dev.device, [&] {
        if (cudaFuncSetAttribute(matvec_kernel<WT, SU, FUSE, SPLIT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 dev.max_smem_optin) != cudaSuccess)
            return QMM_E_CUDA;
        // all of the SM's unified memory as shared memory, so that two small CTAs fit
        if (cudaFuncSetAttribute(matvec_kernel<WT, SU, FUSE, SPLIT>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 (int)cudaSharedmemCarveoutMaxShared) != cudaSuccess)
            return QMM_E_CUDA;
        return QMM_OK;
    });
    if (ast != QMM_OK) return ast;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.grid);
    cfg.blockDim = dim3((unsigned)(p.nw * 32));
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, matvec_kernel<WT, SU, FUSE, SPLIT>, set, (const uint8_t*)xq, x,
                                             (uint8_t*)xq_out, (int)K, p.lpr, p.pieces, p.piece_units, p.item_segs,
                                             p.depth, p.slot_bytes, p.part_off, p.act_bytes, pdl ? 1 : 0);
    return e == cudaSuccess ? QMM_OK : QMM_E_CUDA;
}

template <int WT, bool SU, int FUSE>
static qmm_status launch_matvec_su(const MatSet& set, const void* xq, const float* x, void* xq_out, int64_t K,
                                   const MatvecPlan& p, const DeviceInfo& dev, cudaStream_t stream, bool pdl) {
    if (p.pieces > 1) return launch_matvec_k<WT, SU, FUSE, true>(set, xq, x, xq_out, K, p, dev, stream, pdl);
    return launch_matvec_k<WT, SU, FUSE, false>(set, xq, x, xq_out, K, p, dev, stream, pdl);
}

// G matrices W[g] (N[g] rows each) against one activation row.  x == nullptr:
// multiply the quantized row xq.  Otherwise quantize x in the kernel (xq then
// names where CTA 0 stores the quantized row, or is null).
template <int WT>
static qmm_status launch_matvec(const void* const* W, const int64_t* N, float* const* y, int G, const void* xq,
                                const float* x, int64_t K, cudaStream_t stream, bool pdl, const float* gamma,
                                float eps) {
    if (G < 1 || G > kMaxGroup) return QMM_E_SHAPE;
    DeviceInfo dev;
    qmm_status st = current_device(&dev);
    if (st != QMM_OK) return st;
    MatvecPlan p;
    MatSet set = {};
    const bool fuse = x != nullptr;
    st = plan_matvec<WT>(N, G, K, dev, fuse, fuse && gamma != nullptr, &p, set.cta_end);
    if (st != QMM_OK) return st;
    set.G = G;
    set.gamma = fuse ? gamma : nullptr;
    set.eps = eps;
    set.norm_off = p.norm_off;
    for (int g = 0; g < G; g++) {
        set.W[g] = (const uint8_t*)W[g];
        set.y[g] = y[g];
        set.N[g] = (int)N[g];
    }
    if (fuse && gamma != nullptr) {  // RMSNorm, quantize and multiply
        if constexpr (has_su<WT>()) {
            if (p.su) return launch_matvec_su<WT, true, 2>(set, nullptr, x, (void*)xq, K, p, dev, stream, pdl);
        }
        return launch_matvec_su<WT, false, 2>(set, nullptr, x, (void*)xq, K, p, dev, stream, pdl);
    }
    if (fuse) {  // quantize and multiply
        if constexpr (has_su<WT>()) {
            if (p.su) return launch_matvec_su<WT, true, 1>(set, nullptr, x, (void*)xq, K, p, dev, stream, pdl);
        }
        return launch_matvec_su<WT, false, 1>(set, nullptr, x, (void*)xq, K, p, dev, stream, pdl);
    }
    if constexpr (has_su<WT>()) {
        if (p.su) return launch_matvec_su<WT, true, 0>(set, xq, nullptr, nullptr, K, p, dev, stream, pdl);
    }
    return launch_matvec_su<WT, false, 0>(set, xq, nullptr, nullptr, K, p, dev, stream, pdl);
}

// Public calls require 16-byte aligned bases; internal per-token calls pass rows
// of a larger buffer, which the kernel accepts at their natural alignment (W
// 16 bytes for the bulk copies, an activation row 2 bytes, y 4 bytes; an f32
// row x to quantize in the kernel 16 bytes).
static qmm_status matvec_group_checked(int wt, int G, const void* const* W, const int64_t* N, float* const* y,
                                       const void* xq, const float* x, int64_t K, cudaStream_t stream, bool pdl,
                                       bool public_call, const float* gamma = nullptr, float eps = 0.0f) {
    if (G < 1 || G > kMaxGroup) return QMM_E_SHAPE;
    if (!W || !N || !y || (!xq && !x)) return QMM_E_NULL;
    for (int g = 0; g < G; g++) {
        if (!W[g] || !y[g]) return QMM_E_NULL;
        qmm_status st = check_shape(wt, 1, N[g], K);
        if (st != QMM_OK) return st;
        if (public_call && (!aligned16(W[g]) || !aligned16(y[g]))) return QMM_E_ALIGN;
        if (!aligned16(W[g]) || ((uintptr_t)y[g] & 3u)) return QMM_E_ALIGN;
    }
    if (public_call && !aligned16(xq)) return QMM_E_ALIGN;
    if (((uintptr_t)xq & 1u) || !aligned16(x) || !aligned16(gamma)) return QMM_E_ALIGN;
    switch (wt) {
    case QMM_Q4_0: return launch_matvec<QMM_Q4_0>(W, N, y, G, xq, x, K, stream, pdl, gamma, eps);
    case QMM_Q8_0: return launch_matvec<QMM_Q8_0>(W, N, y, G, xq, x, K, stream, pdl, gamma, eps);
    case QMM_Q4_K: return launch_matvec<QMM_Q4_K>(W, N, y, G, xq, x, K, stream, pdl, gamma, eps);
    case QMM_Q6_K: return launch_matvec<QMM_Q6_K>(W, N, y, G, xq, x, K, stream, pdl, gamma, eps);
    case QMM_Q2_K: return launch_matvec<QMM_Q2_K>(W, N, y, G, xq, x, K, stream, pdl, gamma, eps);
    case QMM_Q4_1: return launch_matvec<QMM_Q4_1>(W, N, y, G, xq, x, K, stream, pdl, gamma, eps);
    case QMM_Q5_0: return launch_matvec<QMM_Q5_0>(W, N, y, G, xq, x, K, stream, pdl, gamma, eps);
    case QMM_Q5_1: return launch_matvec<QMM_Q5_1>(W, N, y, G, xq, x, K, stream, pdl, gamma, eps);
    case QMM_Q5_K: return launch_matvec<QMM_Q5_K>(W, N, y, G, xq, x, K, stream, pdl, gamma, eps);
    default: return QMM_E_TYPE;
    }
}

static qmm_status matvec_checked(int wt, const void* W, const void* xq, const float* x, float* y, int64_t N,
                                 int64_t K, cudaStream_t stream, bool pdl, bool public_call) {
    return matvec_group_checked(wt, 1, &W, &N, &y, xq, x, K, stream, pdl, public_call);
}

qmm_status matvec_dispatch(int wt, const void* W, const void* xq, float* y, int64_t N, int64_t K, cudaStream_t stream,
                           bool pdl) {
    return matvec_checked(wt, W, xq, nullptr, y, N, K, stream, pdl, false);
}

// Quantize one f32 row x and multiply, in one launch; the quantized row is also
// stored to xq_out (when not null).  Fails with QMM_E_SHAPE when the row does not
// fit the kernel's shared memory, so the caller can quantize separately instead.
qmm_status matvec_fused_dispatch(int wt, const void* W, const float* x, void* xq_out, float* y, int64_t N, int64_t K,
                                 cudaStream_t stream, bool pdl) {
    if (!x) return QMM_E_NULL;
    return matvec_checked(wt, W, xq_out, x, y, N, K, stream, pdl, false);
}

// The same for G matrices sharing the row (xq_out as above).
qmm_status matvec_group_fused_dispatch(int wt, int G, const void* const* W, const int64_t* N, float* const* y,
                                       const float* x, void* xq_out, int64_t K, cudaStream_t stream, bool pdl) {
    if (!x) return QMM_E_NULL;
    return matvec_group_checked(wt, G, W, N, y, xq_out, x, K, stream, pdl, false);
}

// The same with the row RMSNormed by gamma (eps) before it is quantized.
qmm_status matvec_group_norm_dispatch(int wt, int G, const void* const* W, const int64_t* N, float* const* y,
                                      const float* x, const float* gamma, float eps, void* xq_out, int64_t K,
                                      cudaStream_t stream, bool pdl) {
    if (!x || !gamma) return QMM_E_NULL;
    return matvec_group_checked(wt, G, W, N, y, xq_out, x, K, stream, pdl, false, gamma, eps);
}

// G matrices against one quantized row (internal: alignment as for per-token rows).
qmm_status matvec_group_dispatch(int wt, int G, const void* const* W, const int64_t* N, float* const* y,
                                 const void* xq, int64_t K, cudaStream_t stream, bool pdl) {
    return matvec_group_checked(wt, G, W, N, y, xq, nullptr, K, stream, pdl, false);
}

template <int WT>
static qmm_status launch_blocksums(const void* W, const void* xq, int32_t* s, int64_t M, int64_t N, int64_t K,
                                   cudaStream_t stream) {
    using F = Fmt<WT>;
    DeviceInfo dev;
    qmm_status st = current_device(&dev);
    if (st != QMM_OK) return st;
    const uint64_t rb = (uint64_t)(K / F::BV) * F::BB;
    const uint32_t act = 128u + act_region_bytes(F::ACT, (int)K);
    int rows = (int)(16384 / rb);
    if (rows < 1) rows = 1;
    if (rows > 64) rows = 64;
    const uint64_t smem = act + align_up((uint32_t)(rows * rb + 48), 128u);
    if (smem > (uint64_t)dev.max_smem_optin) return QMM_E_SHAPE;
    if (cudaFuncSetAttribute(blocksums_kernel<WT>, cudaFuncAttributeMaxDynamicSharedMemorySize, dev.max_smem_optin) !=
        cudaSuccess)
        return QMM_E_CUDA;
    const dim3 grid((unsigned)((N + rows - 1) / rows), (unsigned)M);
    if (M > 65535) return QMM_E_SHAPE;
    blocksums_kernel<WT><<<grid, kThreads, (size_t)smem, stream>>>((const uint8_t*)W, (const uint8_t*)xq, s, (int)N,
                                                                   (int)K, rows, act);
    return launch_status();
}

}  // namespace qmm

using namespace qmm;

extern "C" {

qmm_status qmm_matvec_q4_0(const void* W, const void* xq, float* y, int64_t N, int64_t K, qmm_stream_t stream) {
    return matvec_checked(QMM_Q4_0, W, xq, nullptr, y, N, K, (cudaStream_t)stream, true, true);
}
qmm_status qmm_matvec_q8_0(const void* W, const void* xq, float* y, int64_t N, int64_t K, qmm_stream_t stream) {
    return matvec_checked(QMM_Q8_0, W, xq, nullptr, y, N, K, (cudaStream_t)stream, true, true);
}
qmm_status qmm_matvec_q4_K(const void* W, const void* xq, float* y, int64_t N, int64_t K, qmm_stream_t stream) {
    return matvec_checked(QMM_Q4_K, W, xq, nullptr, y, N, K, (cudaStream_t)stream, true, true);
}
qmm_status qmm_matvec_q6_K(const void* W, const void* xq, float* y, int64_t N, int64_t K, qmm_stream_t stream) {
    return matvec_checked(QMM_Q6_K, W, xq, nullptr, y, N, K, (cudaStream_t)stream, true, true);
}
qmm_status qmm_matvec_q2_K(const void* W, const void* xq, float* y, int64_t N, int64_t K, qmm_stream_t stream) {
    return matvec_checked(QMM_Q2_K, W, xq, nullptr, y, N, K, (cudaStream_t)stream, true, true);
}
qmm_status qmm_matvec_q4_1(const void* W, const void* xq, float* y, int64_t N, int64_t K, qmm_stream_t stream) {
    return matvec_checked(QMM_Q4_1, W, xq, nullptr, y, N, K, (cudaStream_t)stream, true, true);
}
qmm_status qmm_matvec_q5_0(const void* W, const void* xq, float* y, int64_t N, int64_t K, qmm_stream_t stream) {
    return matvec_checked(QMM_Q5_0, W, xq, nullptr, y, N, K, (cudaStream_t)stream, true, true);
}
qmm_status qmm_matvec_q5_1(const void* W, const void* xq, float* y, int64_t N, int64_t K, qmm_stream_t stream) {
    return matvec_checked(QMM_Q5_1, W, xq, nullptr, y, N, K, (cudaStream_t)stream, true, true);
}
qmm_status qmm_matvec_q5_K(const void* W, const void* xq, float* y, int64_t N, int64_t K, qmm_stream_t stream) {
    return matvec_checked(QMM_Q5_K, W, xq, nullptr, y, N, K, (cudaStream_t)stream, true, true);
}

qmm_status qmm_blocksums(int wtype, const void* W, const void* xq, int32_t* s, int64_t M, int64_t N, int64_t K,
                         qmm_stream_t stream) {
    if (act_type_of(wtype) < 0) return QMM_E_TYPE;
    if (!W || !xq || !s) return QMM_E_NULL;
    qmm_status st = check_shape(wtype, M, N, K);
    if (st != QMM_OK) return st;
    if (!aligned16(W) || !aligned16(xq) || !aligned16(s)) return QMM_E_ALIGN;
    cudaStream_t cs = (cudaStream_t)stream;
    switch (wtype) {
    case QMM_Q4_0: return launch_blocksums<QMM_Q4_0>(W, xq, s, M, N, K, cs);
    case QMM_Q8_0: return launch_blocksums<QMM_Q8_0>(W, xq, s, M, N, K, cs);
    case QMM_Q4_K: return launch_blocksums<QMM_Q4_K>(W, xq, s, M, N, K, cs);
    case QMM_Q6_K: return launch_blocksums<QMM_Q6_K>(W, xq, s, M, N, K, cs);
    case QMM_Q2_K: return launch_blocksums<QMM_Q2_K>(W, xq, s, M, N, K, cs);
    case QMM_Q4_1: return launch_blocksums<QMM_Q4_1>(W, xq, s, M, N, K, cs);
    case QMM_Q5_0: return launch_blocksums<QMM_Q5_0>(W, xq, s, M, N, K, cs);
    case QMM_Q5_1: return launch_blocksums<QMM_Q5_1>(W, xq, s, M, N, K, cs);
    case QMM_Q5_K: return launch_blocksums<QMM_Q5_K>(W, xq, s, M, N, K, cs);
    default: return QMM_E_TYPE;
    }
}

unsigned qmm_internal_matvec_error(int clear) {
    unsigned v = 0;
    cudaMemcpyFromSymbol(&v, g_matvec_error, sizeof(v));
    if (clear) {
        const unsigned z = 0;
        cudaMemcpyToSymbol(g_matvec_error, &z, sizeof(z));
    }
    return v;
}

}  // extern "C"
