// matmul.cu -- the prefill matmul Y[M][N] for Q4_0 or Q8_0 weights x Q8_0
// activations, M tokens at once, on the 5th-generation tensor cores.
//
// Y[t][o] = sum_b d_w[o,b] * d_x[t,b] * isum[t,o,b] ([krafla] "Architecture",
// Batched prompt prefill; [kvad] "Batched prefill, and i8mm"): the weights are
// read once per tile of 128 tokens instead of once per token.
//
// sm_103a has no int8 tensor-core MMA (ptxas rejects tcgen05.mma .kind::i8 for
// this target), so the integer codes go through .kind::f16 with fp16 operands:
// every Q4_0 code (-8..7) and Q8_0 code (-128..127) is an exact fp16 value, all
// products are exact, and each 32-wide block's sum (|sum| <= 32*128*128 < 2^24) is
// exact in the fp32 accumulator -- the MMA computes the same integer isum the
// scalar kernel does ([minfer] s3.2: the integer dot is exact; [ggml] s2).
// Each block's sum is then folded into an fp32 accumulator once, scaled by
// d_w * d_x, exactly as the pages' kernels fold per block.
//
// One CTA per output tile of 128 weight rows x 128 tokens, 26 warps:
//   warp 24  producer: 2-D TMA loads of the raw weight bytes (128 rows x 8 blocks)
//            and the raw activation bytes (128 tokens x 8 blocks) into a ring of
//            raw stages; also owns the tensor-memory allocation
//   warp 25  MMA issuer: per block, two tcgen05.mma (K = 16 each) with the
//            weight operand read from TMEM and the activation operand from shared
//            memory, into one of three 128-column TMEM accumulators; one
//            tcgen05.commit frees the operand slot, another hands over the sums
//   warps 16-19 weight converters: each thread turns its row's blocks into fp16
//            operands and stores them straight into its TMEM lane (tcgen05.st;
//            warp % 4 is that lane quadrant), plus the f32 scale
//   warps 20-23 activation converters: each thread turns its token's blocks
//            into fp16 operands in the UMMA K-major core-matrix layout (8 rows x
//            16 bytes per core matrix) in shared memory, plus the f32 scale
//   warps 0-15 epilogue: tcgen05.ld of each block's exact sums (32 tokens of one
//            weight row per thread), y += v * (d_w*d_x) in registers in block
//            order, then the token-major store
// The weight operand never passes through shared memory, so the tensor core
// reads only the activation tile from it.  All waits are bounded; a timeout
// records QMM_E_TIMEOUT, every warp still reaches the end, and TMEM is freed.
#include <cuda.h>
#include <mutex>

#include "qmm_device.cuh"
#include "qmm_host.h"
#include "tc_device.cuh"

namespace qmm {

static __device__ unsigned int g_matmul_error = 0;

qmm_status matvec_dispatch(int wt, const void* W, const void* xq, float* y, int64_t N, int64_t K, cudaStream_t stream,
                           bool pdl);
qmm_status matmul_kq_launch(int wt, const void* W, const void* xq, float* Y, int64_t M, int64_t N, int64_t K,
                            cudaStream_t stream, bool pdl);
bool kq_uses_tensor_cores(int wt, int64_t M, int64_t K);

namespace mm {

constexpr int BM = 128;            // weight rows per tile (MMA M, TMEM lanes)
constexpr int BN = 128;            // tokens per tile (MMA N, TMEM columns per accumulator)
constexpr int KB = 8;              // Q blocks per raw stage (256 K values)
constexpr int RAW_STAGES = 2;
constexpr int S_BUFS = 3;          // per-block sum accumulators in TMEM, 128 columns each
constexpr int OP_SLOTS = 4;        // operand slots: weights in TMEM (16 columns), activations in shared memory
constexpr int A_COL0 = S_BUFS * BN;  // TMEM column of weight operand slot 0 (after the accumulators)
constexpr int TMEM_COLS = 512;
static_assert(A_COL0 + OP_SLOTS * 16 <= TMEM_COLS, "TMEM layout");
// One tcgen05.commit per block signals "the MMAs of block b are done" on
// mma_done[b % DONE_RING]: the epilogue waits for it to read block b's sums, the
// converters to reuse block b's operand slot for block b + OP_SLOTS.  A barrier
// is reused DONE_RING blocks later, which neither waiter can reach first: the
// MMAs of block b + DONE_RING need the epilogue to have released block
// b + DONE_RING - S_BUFS > b, and the converters' operands of that block.
constexpr int DONE_RING = 8;
static_assert(DONE_RING >= S_BUFS + 3 && DONE_RING >= OP_SLOTS + 2 && (DONE_RING & (DONE_RING - 1)) == 0,
              "mma_done ring");
constexpr int X_RAW = BN * KB * 34;   // 34816
constexpr int OP_B = BN * 32 * 2;     // 8192: fp16 activations of one block
constexpr int NUM_EPI_WARPS = 16, NUM_W_WARPS = 4, NUM_X_WARPS = 4;
constexpr int NUM_CONV_WARPS = NUM_W_WARPS + NUM_X_WARPS;
// Warps 0-15: epilogue (warp % 4 is the TMEM lane quadrant it may read, warp / 4
// its 32 tokens); 16-19: weight converters (warp % 4 = the lane quadrant of the
// 32 rows each writes into TMEM); 20-23: activation converters; 24: TMA producer
// (and the TMEM allocation); 25: MMA issuer.
// With the activation pre-pass (XP) the activation converters are gone and the
// producer also copies each chunk's prepared operands: 22 warps.
constexpr int W0 = NUM_EPI_WARPS, X0 = W0 + NUM_W_WARPS;
template <bool XP>
struct Roles {
    static constexpr int TMA_WARP = X0 + (XP ? 0 : NUM_X_WARPS), MMA_WARP = TMA_WARP + 1;
    static constexpr int THREADS = (MMA_WARP + 1) * 32;  // 832, or 704 with the pre-pass
    static constexpr int CONV_WARPS = NUM_W_WARPS + (XP ? 0 : NUM_X_WARPS);  // arrivals per slot / stage
};

// Weight block bytes of the 32-value formats (Q4_0 18, Q8_0 34, Q4_1 20, Q5_0 22, Q5_1 24).
__host__ __device__ constexpr int block_bytes32(int wt) {
    return wt == QMM_Q8_0 ? 34 : wt == QMM_Q4_1 ? 20 : wt == QMM_Q5_0 ? 22 : wt == QMM_Q5_1 ? 24 : 18;
}

// Shared memory layout per weight format (offsets from the 1024-byte aligned
// dynamic shared memory base): the raw stages, the activation operand slots and
// the per-block scales.  Q4_1 and Q5_1 also carry each row's m_w and each
// token's d_x * sum(a) per block, for the min term.
template <int WT, bool XP = false>
struct Lay {
    static constexpr int WB = block_bytes32(WT);
    static constexpr bool HAS_MIN = WT == QMM_Q4_1 || WT == QMM_Q5_1;
    // Blocks of scales in flight.  A slot is rewritten for block b by a converter
    // that has waited for the MMAs of block b - OP_SLOTS, which the MMA issuer
    // started only after the epilogue released the sums of block
    // b - OP_SLOTS - S_BUFS; the epilogue works in block order, so it had
    // finished every read of block b - OP_SLOTS - S_BUFS - 1 and earlier.
    static constexpr int SC_SLOTS = 16;
    static_assert(SC_SLOTS >= OP_SLOTS + S_BUFS + 1, "scale slots must outlive the epilogue's reads");
    static constexpr int W_RAW = BM * KB * WB;
    static constexpr int RAW_BYTES = W_RAW + (XP ? 0 : X_RAW);
    // XP: a chunk of prepared activation operands, as the pre-pass writes it and
    // one bulk copy brings it in: KB blocks of fp16 codes (the core-matrix layout
    // the MMA reads), each block's d_x for the 128 tokens, and (min formats) each
    // block's d_x * sum(a)
    static constexpr int XPS = KB * OP_B + KB * BN * 4 + (HAS_MIN ? KB * BN * 4 : 0);
    static constexpr int OFF_RAW = 0;
    static constexpr int OFF_XP = OFF_RAW + RAW_STAGES * RAW_BYTES;  // XP: RAW_STAGES chunks of XPS
    static constexpr int OFF_OPB = OFF_XP + (XP ? RAW_STAGES * XPS : 0);
    static constexpr int OFF_SCW = OFF_OPB + (XP ? 0 : OP_SLOTS * OP_B);
    static constexpr int OFF_SCX = OFF_SCW + SC_SLOTS * BM * 4;
    static constexpr int OFF_SCM = OFF_SCX + SC_SLOTS * BN * 4;            // m_w per row (min formats)
    static constexpr int OFF_SCS = OFF_SCM + (HAS_MIN ? SC_SLOTS * BM * 4 : 0);  // d_x * sum(a) per token
    static constexpr int OFF_BAR = OFF_SCS + (HAS_MIN ? SC_SLOTS * BN * 4 : 0);
    // barriers: raw_full[2] raw_empty[2] op_full[4] mma_done[8] acc_empty[3] x_full[2] x_empty[2]
    static constexpr int NBARS = 2 * RAW_STAGES + OP_SLOTS + DONE_RING + S_BUFS + 2 * RAW_STAGES;
    static constexpr int OFF_TMEM = OFF_BAR + NBARS * 8;
    static constexpr int SMEM_BYTES = OFF_TMEM + 16;
};
static_assert(Lay<QMM_Q4_0>::SMEM_BYTES <= 232448 && Lay<QMM_Q8_0>::SMEM_BYTES <= 232448 &&
                  Lay<QMM_Q4_1>::SMEM_BYTES <= 232448 && Lay<QMM_Q5_0>::SMEM_BYTES <= 232448 &&
                  Lay<QMM_Q5_1>::SMEM_BYTES <= 232448,
              "prefill smem");
static_assert(Lay<QMM_Q4_0, true>::SMEM_BYTES <= 232448 && Lay<QMM_Q8_0, true>::SMEM_BYTES <= 232448 &&
                  Lay<QMM_Q4_1, true>::SMEM_BYTES <= 232448 && Lay<QMM_Q5_0, true>::SMEM_BYTES <= 232448 &&
                  Lay<QMM_Q5_1, true>::SMEM_BYTES <= 232448,
              "prefill smem (pre-pass)");
static_assert(Lay<QMM_Q4_0, true>::OFF_XP % 128 == 0 && Lay<QMM_Q8_0, true>::OFF_XP % 128 == 0 &&
                  Lay<QMM_Q4_1, true>::OFF_XP % 128 == 0 && Lay<QMM_Q5_0, true>::OFF_XP % 128 == 0 &&
                  Lay<QMM_Q5_1, true>::OFF_XP % 128 == 0 && Lay<QMM_Q4_1, true>::XPS % 128 == 0 &&
                  Lay<QMM_Q4_0, true>::XPS % 128 == 0,
              "operand tiles need 128-byte alignment");

struct Bars {
    uint32_t base;
    __device__ uint32_t raw_full(int i) const { return base + 8u * i; }
    __device__ uint32_t raw_empty(int i) const { return base + 8u * (RAW_STAGES + i); }
    // operand slot i written by the converters
    __device__ uint32_t op_full(int i) const { return base + 8u * (2 * RAW_STAGES + i); }
    // the MMAs of block b done (one tcgen05.commit): barrier b % DONE_RING, phase b / DONE_RING
    __device__ uint32_t mma_done(int b) const { return base + 8u * (2 * RAW_STAGES + OP_SLOTS + (b & (DONE_RING - 1))); }
    // accumulator i read into registers by every epilogue warp
    __device__ uint32_t acc_empty(int i) const { return base + 8u * (2 * RAW_STAGES + OP_SLOTS + DONE_RING + i); }
    // XP: the prepared chunk in stage i landed / was used by the MMAs and the epilogue
    __device__ uint32_t x_full(int i) const {
        return base + 8u * (2 * RAW_STAGES + OP_SLOTS + DONE_RING + S_BUFS + i);
    }
    __device__ uint32_t x_empty(int i) const {
        return base + 8u * (3 * RAW_STAGES + OP_SLOTS + DONE_RING + S_BUFS + i);
    }
};

// wait with a time limit; on failure set the error word and the CTA's abort flag.
// The fast path (phase already complete) is a single try_wait.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (mbar_wait_bounded(bar, parity, kWaitLimitNs)) return true;
    atomicOr(&g_matmul_error, kErrTimeout);
    *abort_flag = 1;
    return false;
}

// One block of 32 converted values of a row (fp16 pairs in K order: register c
// holds elements 2c and 2c+1) into its operand slot: weights into this warp's
// TMEM lanes, activations into the K-major core-matrix layout in shared memory.
template <bool IS_W>
__device__ __forceinline__ void put_operand(const uint32_t (&h)[16], uint32_t tmem_a, uint8_t* opb_row) {
    if constexpr (IS_W) {
        tc_fence_after();  // after the wait that freed the slot (its last MMA read it)
        tmem_st16(tmem_a, h);
        tmem_st_wait();
        tc_fence_before();
    } else {
#pragma unroll
        for (int kq = 0; kq < 4; kq++)
            *reinterpret_cast<uint4*>(opb_row + kq * 128) = make_uint4(h[4 * kq], h[4 * kq + 1], h[4 * kq + 2], h[4 * kq + 3]);
        fence_proxy_async_smem();  // the operands are read by the tensor core (async proxy)
    }
}

// The converter loop of one role.  IS_W: weight rows (WT's block layout) into
// TMEM; otherwise Q8_0 tokens into shared memory.  Each thread owns one row or
// token of the tile; per block it waits for the operand slot (freed by the MMAs
// of block b - OP_SLOTS; that also frees the block's scale slot), converts, and
// hands the block to the MMA issuer.
template <int WT, bool IS_W, bool XP>
__device__ __forceinline__ void convert_loop(uint8_t* smem, uint32_t sbase, const Bars& bars, uint32_t tmem, int r,
                                             int nchunks, volatile int* abort_flag) {
    using L = Lay<WT, XP>;
    constexpr int SC_SLOTS = L::SC_SLOTS, RAW_BYTES = L::RAW_BYTES, W_RAW = L::W_RAW;
    constexpr int RB = IS_W ? L::WB : 34;  // raw block bytes of this role
    static_assert(KB % OP_SLOTS == 0 && SC_SLOTS == 2 * KB && DONE_RING == KB,
                  "slot indices are fixed per block of a chunk");
    const int lane = threadIdx.x & 31;
    const uint32_t tmem_row = tmem + ((uint32_t)(r & ~31) << 16) + (uint32_t)A_COL0;  // this warp's lane quadrant
    // this thread's row in the activation operand slots (K-major core matrices)
    uint8_t* const opb_row = smem + L::OFF_OPB + ((r >> 3) * 4) * 128 + (r & 7) * 16;
    float* const scale_row = reinterpret_cast<float*>(smem + (IS_W ? L::OFF_SCW : L::OFF_SCX)) + r;
    float* const mw_row = reinterpret_cast<float*>(smem + L::OFF_SCM) + r;
    float* const asum_row = reinterpret_cast<float*>(smem + L::OFF_SCS) + r;
    // XP: the weight threads also move token r's prepared d_x (and d_x * sum(a)) of
    // each block from the chunk's stage into the scale ring the epilogue reads
    float* const xscale_row = reinterpret_cast<float*>(smem + L::OFF_SCX) + r;
    bool ok = true;
    for (int c = 0; c < nchunks && ok; c++) {
        const int s = c % RAW_STAGES;
        if (!wait_or_abort(bars.raw_full(s), (c / RAW_STAGES) & 1, abort_flag)) break;
        if (XP && IS_W && !__all_sync(0xffffffffu, wait_or_abort(bars.x_full(s), (c / RAW_STAGES) & 1, abort_flag)))
            break;
        const float* const xstage = reinterpret_cast<const float*>(smem + L::OFF_XP + s * L::XPS + KB * OP_B) + r;
        const uint8_t* row = smem + L::OFF_RAW + s * RAW_BYTES + (IS_W ? 0 : W_RAW) + r * (KB * RB);
        // the row's 8 blocks, read as two windows of 4 blocks from the 16-byte boundary at or
        // below each window's first byte (rows of 8 blocks are 16-byte multiples)
#pragma unroll
        for (int hw = 0; hw < 2 && ok; hw++) {
            const int start = 4 * RB * hw, base16 = start & ~15, off0 = start - base16;
            constexpr int NV = (4 * RB + 15 + 15) / 16;  // 16-byte loads covering a window at any offset
            uint32_t raw[4 * NV + 1];
            raw[4 * NV] = 0;
            const int nv = (off0 + 4 * RB + 15) / 16;
            const uint4* src = reinterpret_cast<const uint4*>(row + base16);
#pragma unroll
            for (int i = 0; i < NV; i++) {
                const uint4 v = i < nv ? src[i] : make_uint4(0u, 0u, 0u, 0u);
                raw[4 * i] = v.x; raw[4 * i + 1] = v.y; raw[4 * i + 2] = v.z; raw[4 * i + 3] = v.w;
            }
#pragma unroll
            for (int lq = 0; lq < KB / 2; lq++) {
                // block b = c * KB + kb of the chunk: operand slot kb % OP_SLOTS, scale slot
                // (c & 1) * KB + kb; its slot was last used by block b - OP_SLOTS, whose
                // mma_done barrier is (kb - OP_SLOTS) mod KB, in phase c (or c - 1)
                const int kb = 4 * hw + lq, os = kb % OP_SLOTS, ssl = (c & 1) * KB + kb;
                const int kprev = kb - OP_SLOTS;  // the previous user's block within its chunk
                const bool freed =
                    (c == 0 && kprev < 0) ||
                    wait_or_abort(bars.mma_done((kprev + KB) % KB), (kprev < 0 ? c - 1 : c) & 1, abort_flag);
                if (!__all_sync(0xffffffffu, freed)) {  // warp-uniform: the TMEM store below is warp-collective
                    ok = false;
                    break;
                }
                const int off = off0 + RB * lq;  // the block's first byte in the window
                auto word_at = [&](int o) -> uint32_t {
                    return (o % 4 == 0) ? raw[o / 4] : __funnelshift_r(raw[o / 4], raw[o / 4 + 1], 8 * (o % 4));
                };
                uint32_t h[16];
                if constexpr (IS_W && WT != QMM_Q8_0) {
                    // Q4_0: d, qs@2; Q4_1: d, m, qs@4; Q5_0: d, qh@2, qs@6; Q5_1: d, m, qh@4, qs@8;
                    // element j is the low nibble of qs[j], element j+16 the high one, and bit e of
                    // qh is element e's fifth bit
                    constexpr int OFF_Q = WT == QMM_Q4_0 ? 2 : WT == QMM_Q4_1 ? 4 : WT == QMM_Q5_0 ? 6 : 8;
                    constexpr int OFF_H = WT == QMM_Q5_0 ? 2 : 4;
                    constexpr bool FIVE = WT == QMM_Q5_0 || WT == QMM_Q5_1;
                    // fp16 bits of (1024 + code) minus 1032 (Q4_0: code - 8), 1040 (Q5_0: code - 16)
                    // or 1024 (Q4_1, Q5_1: the code itself)
                    constexpr uint32_t magic =
                        WT == QMM_Q4_0 ? 0x64086408u : WT == QMM_Q5_0 ? 0x64106410u : 0x64006400u;
                    const uint32_t dm = word_at(off);  // d in the low half, m (Q4_1, Q5_1) in the high half
                    const uint32_t qh = FIVE ? word_at(off + OFF_H) : 0u;
                    uint32_t lo[4], hi[4];
#pragma unroll
                    for (int i = 0; i < 4; i++) {
                        const uint32_t q = word_at(off + OFF_Q + 4 * i);
                        lo[i] = q & 0x0F0F0F0Fu;
                        hi[i] = (q >> 4) & 0x0F0F0F0Fu;
                        if (FIVE) {
                            lo[i] |= spread4(qh >> (4 * i)) << 4;
                            hi[i] |= spread4(qh >> (16 + 4 * i)) << 4;
                        }
                    }
#pragma unroll
                    for (int kq = 0; kq < 4; kq++) {  // elements 8kq..8kq+7
                        const uint32_t w0 = kq < 2 ? lo[2 * kq] : hi[2 * (kq - 2)];
                        const uint32_t w1 = kq < 2 ? lo[2 * kq + 1] : hi[2 * (kq - 2) + 1];
                        h[4 * kq] = h2_sub(bytes_to_h2(w0, 0x5140), magic);
                        h[4 * kq + 1] = h2_sub(bytes_to_h2(w0, 0x7362), magic);
                        h[4 * kq + 2] = h2_sub(bytes_to_h2(w1, 0x5140), magic);
                        h[4 * kq + 3] = h2_sub(bytes_to_h2(w1, 0x7362), magic);
                    }
                    scale_row[ssl * BM] = h2f(dm & 0xFFFFu);
                    if (L::HAS_MIN) mw_row[ssl * BM] = h2f(dm >> 16);
                } else {
                    // a Q8_0 block (activation token or Q8_0 weight row): f16 d, 32 int8 codes
                    const uint32_t dbits = word_at(off) & 0xFFFFu;
                    const uint32_t m128 = 0x64806480u;  // (1152, 1152): 1024 + (a + 128) - 1152 = a
                    int asum = 0;  // sum of the block's codes (min formats: the token's m_w term)
#pragma unroll
                    for (int kq = 0; kq < 4; kq++) {  // elements 8kq..8kq+7: code words 2kq, 2kq+1
                        const uint32_t c0 = word_at(off + 2 + 8 * kq), c1 = word_at(off + 6 + 8 * kq);
                        if (!IS_W && L::HAS_MIN) asum = __dp4a((int)c1, 0x01010101, __dp4a((int)c0, 0x01010101, asum));
                        const uint32_t w0 = c0 ^ 0x80808080u, w1 = c1 ^ 0x80808080u;
                        h[4 * kq] = h2_sub(bytes_to_h2(w0, 0x5140), m128);
                        h[4 * kq + 1] = h2_sub(bytes_to_h2(w0, 0x7362), m128);
                        h[4 * kq + 2] = h2_sub(bytes_to_h2(w1, 0x5140), m128);
                        h[4 * kq + 3] = h2_sub(bytes_to_h2(w1, 0x7362), m128);
                    }
                    scale_row[ssl * BN] = h2f(dbits);
                    if (!IS_W && L::HAS_MIN) asum_row[ssl * BN] = h2f(dbits) * (float)asum;
                }
                if (XP && IS_W) {  // token r's prepared scales of this block into the ring
                    xscale_row[ssl * BN] = xstage[kb * BN];
                    if (L::HAS_MIN) asum_row[ssl * BN] = xstage[(KB + kb) * BN];
                }
                put_operand<IS_W>(h, tmem_row + (uint32_t)(os * 16), opb_row + os * OP_B);
                __syncwarp();
                if (lane == 0) mbar_arrive(bars.op_full(os));
            }
        }
        // The raw stage goes back to the producer only once every value read from it
        // has been used: released right after the loads, the next chunk's TMA was seen
        // to overwrite a window whose loads a converter had just issued.
        __syncwarp();
        if (lane == 0) mbar_arrive(bars.raw_empty(s));
        if (XP && IS_W && lane == 0) mbar_arrive(bars.x_empty(s));  // the chunk's scales are copied
    }
}

// ------------------------------------------------------------------ the activation pre-pass
// Every CTA of a token tile converts the same Q8_0 rows, so with a workspace they
// are converted once: token tile ty's chunk c (blocks 8c .. 8c + 7) becomes
// Lay<WT, true>::XPS bytes -- per block the fp16 codes of the tile's 128 tokens in
// the core-matrix layout the MMA reads, then per block the f32 d_x of the 128
// tokens, then (MIN) per block d_x * sum(a).  CTA (b, ty) writes block b's parts,
// one thread per token; tokens past M get zeros.  The conversions are the in-kernel converter's, so
// the operands are the same bits.
template <bool MIN>
__global__ void __launch_bounds__(BN) q8_0_xprep_kernel(const uint8_t* __restrict__ xq, uint8_t* __restrict__ xp,
                                                        int M, int nchunks, int chunk_bytes, int pdl) {
    if (pdl) pdl_launch_dependents();
    if (pdl) pdl_wait();  // the rows come from the previous kernel
    const int r = threadIdx.x, b = blockIdx.x, ty = blockIdx.y;
    const int c = b / KB, kb = b % KB;
    const int t = ty * BN + r;
    const bool real = t < M && QMM_IN_BOUNDS(g_matmul_error, t, M);
    uint8_t* out = xp + ((size_t)ty * nchunks + c) * chunk_bytes;
    const uint32_t m128 = 0x64806480u;  // (1152, 1152): 1024 + (a + 128) - 1152 = a
    {
        // 34-byte blocks are 2-byte aligned: 16-bit loads
        const unsigned short* p =
            reinterpret_cast<const unsigned short*>(xq + ((size_t)(real ? t : 0) * nchunks * KB + (size_t)b) * 34);
        const uint32_t dbits = real ? p[0] : 0u;
        int asum = 0;
#pragma unroll
        for (int kq = 0; kq < 4; kq++) {  // elements 8kq..8kq+7
            const uint32_t c0 = real ? ((uint32_t)p[1 + 4 * kq] | ((uint32_t)p[2 + 4 * kq] << 16)) : 0u;
            const uint32_t c1 = real ? ((uint32_t)p[3 + 4 * kq] | ((uint32_t)p[4 + 4 * kq] << 16)) : 0u;
            if (MIN) asum = __dp4a((int)c1, 0x01010101, __dp4a((int)c0, 0x01010101, asum));
            const uint32_t w0 = c0 ^ 0x80808080u, w1 = c1 ^ 0x80808080u;
            const uint4 v = make_uint4(h2_sub(bytes_to_h2(w0, 0x5140), m128), h2_sub(bytes_to_h2(w0, 0x7362), m128),
                                       h2_sub(bytes_to_h2(w1, 0x5140), m128), h2_sub(bytes_to_h2(w1, 0x7362), m128));
            *reinterpret_cast<uint4*>(out + kb * OP_B + ((r >> 3) * 4 + kq) * 128 + (r & 7) * 16) = v;
        }
        float* sc = reinterpret_cast<float*>(out + KB * OP_B) + kb * BN + r;
        sc[0] = h2f(dbits);
        if (MIN) sc[KB * BN] = h2f(dbits) * (float)asum;
    }
}

// XP: the activation operands come prepared by q8_0_xprep_kernel (xp, one chunk
// of XPS bytes per token tile and 8 blocks); otherwise xmap's raw Q8_0 rows are
// converted here.
template <int WT, bool XP>
__global__ void __launch_bounds__(Roles<XP>::THREADS, 1)
    matmul_q_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap xmap,
                    const uint8_t* __restrict__ xp, float* __restrict__ Y, int M, int N, int K, int pdl) {
    if (pdl) pdl_launch_dependents();
    // used directly (not re-aligned by integer arithmetic) so that the compiler
    // keeps every access in the shared state space
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sbase = smem_u32(smem);
    if (sbase & 127u) {  // the TMA destinations and operand tiles need 128-byte alignment
        if (threadIdx.x == 0) atomicOr(&g_matmul_error, kErrTimeout);
        return;
    }
    using L = Lay<WT, XP>;
    using R = Roles<XP>;
    constexpr int TMA_WARP = R::TMA_WARP, MMA_WARP = R::MMA_WARP;
    if (!QMM_IN_BOUNDS(g_matmul_error, L::SMEM_BYTES - 1, dynamic_smem_bytes())) return;  // the layout must fit
    constexpr int SC_SLOTS = L::SC_SLOTS, W_RAW = L::W_RAW, RAW_BYTES = L::RAW_BYTES, WB = L::WB;
    const Bars bars{sbase + L::OFF_BAR};
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_TMEM);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_TMEM + 8);
    const float* scw = reinterpret_cast<const float*>(smem + L::OFF_SCW);
    const float* scx = reinterpret_cast<const float*>(smem + L::OFF_SCX);
    const float* scm = reinterpret_cast<const float*>(smem + L::OFF_SCM);
    const float* scs = reinterpret_cast<const float*>(smem + L::OFF_SCS);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int o0 = blockIdx.x * BM, t0 = blockIdx.y * BN;
    const int nb = K / 32;
    const int nchunks = nb / KB;

    if (threadIdx.x == 0) {
        for (int i = 0; i < RAW_STAGES; i++) {
            mbar_init(bars.raw_full(i), 1);
            mbar_init(bars.raw_empty(i), R::CONV_WARPS);
            mbar_init(bars.x_full(i), 1);
            mbar_init(bars.x_empty(i), 1 + NUM_W_WARPS);  // the chunk's last MMA commit, the scale copies
        }
        for (int i = 0; i < OP_SLOTS; i++) mbar_init(bars.op_full(i), R::CONV_WARPS);
        for (int i = 0; i < DONE_RING; i++) mbar_init(bars.mma_done(i), 1);
        for (int i = 0; i < S_BUFS; i++) mbar_init(bars.acc_empty(i), NUM_EPI_WARPS);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == TMA_WARP) {  // allocate the TMEM accumulators and weight operand slots (whole warp)
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == TMA_WARP) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            if (pdl) pdl_wait();  // the activation comes from the previous kernel
            for (int c = 0; c < nchunks; c++) {
                const int s = c % RAW_STAGES;
                if (c >= RAW_STAGES && !wait_or_abort(bars.raw_empty(s), ((c / RAW_STAGES) - 1) & 1, abort_flag))
                    break;
                const uint32_t dst = sbase + L::OFF_RAW + s * RAW_BYTES;
                mbar_arrive_expect_tx(bars.raw_full(s), RAW_BYTES);
                tma_load_2d(dst, &wmap, c * (KB * WB / 2), o0, bars.raw_full(s));
                if constexpr (XP) {
                    if (c >= RAW_STAGES && !wait_or_abort(bars.x_empty(s), ((c / RAW_STAGES) - 1) & 1, abort_flag))
                        break;
                    // the prepared chunks are gridDim.y token tiles x nchunks
                    if (!QMM_IN_BOUNDS(g_matmul_error, (int64_t)blockIdx.y * nchunks + c, (int64_t)gridDim.y * nchunks))
                        break;
                    // every CTA of this token tile reads the same chunk: no eviction hint
                    mbar_arrive_expect_tx(bars.x_full(s), (uint32_t)L::XPS);
                    bulk_g2s_nohint(sbase + L::OFF_XP + (uint32_t)(s * L::XPS),
                                    xp + ((size_t)blockIdx.y * nchunks + c) * L::XPS, (uint32_t)L::XPS, bars.x_full(s));
                } else {
                    tma_load_2d(dst + W_RAW, &xmap, c * (KB * 34 / 2), t0, bars.raw_full(s));
                }
            }
        }
    } else if (warp == MMA_WARP) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = instr_desc_f16(BM, BN);
            const uint64_t b0 = smem_desc(sbase + L::OFF_OPB, 128, 512);  // slot os adds os * OP_B (>> 4)
            // block b = round * S_BUFS + sb uses accumulator sb; from round 1 on it waits for the
            // release of round - 1, i.e. phase parity (round - 1) & 1 = s_phase ^ 1
            int sb = 0, s_phase = 0;
            for (int b = 0; b < nb; b++) {
                const int os = b & (OP_SLOTS - 1);
                const int xs = (b / KB) % RAW_STAGES, kb = b % KB;  // XP: the chunk's stage, the block in it
                if (XP && kb == 0 && !wait_or_abort(bars.x_full(xs), (b / KB / RAW_STAGES) & 1, abort_flag)) break;
                if (!wait_or_abort(bars.op_full(os), (b / OP_SLOTS) & 1, abort_flag)) break;
                if (b >= S_BUFS && !wait_or_abort(bars.acc_empty(sb), s_phase ^ 1, abort_flag)) break;
                tc_fence_after();
                const uint32_t a = tmem + (uint32_t)(A_COL0 + os * 16);
                const uint64_t bd =
                    XP ? smem_desc(sbase + L::OFF_XP + (uint32_t)(xs * L::XPS + kb * OP_B), 128, 512)
                       : b0 + (uint64_t)(os * (OP_B >> 4));
                const uint32_t d = tmem + (uint32_t)(sb * BN);
                mma_f16_ts(d, a, bd, idesc, 0);                       // K 0..15: columns 0-7, core matrices 0, 1
                mma_f16_ts(d, a + 8, bd + (256 >> 4), idesc, 1);      // K 16..31: columns 8-15, core matrices 2, 3
                mma_commit(bars.mma_done(b));
                if (XP && kb == KB - 1) mma_commit(bars.x_empty(xs));  // the chunk's operands are read
                if (++sb == S_BUFS) {  // the next round of accumulators: wait for the previous round's release
                    sb = 0;
                    s_phase ^= 1;
                }
            }
        }
    } else if (warp >= W0 && warp < X0) {
        // ------------------------------------------------------------ weight converters
        convert_loop<WT, true, XP>(smem, sbase, bars, tmem, (warp & 3) * 32 + lane, nchunks, abort_flag);
    } else if (!XP && warp >= X0 && warp < TMA_WARP) {
        // ------------------------------------------------------------ activation converters
        convert_loop<WT, false, XP>(smem, sbase, bars, tmem, (warp - X0) * 32 + lane, nchunks, abort_flag);
    } else {
        // ------------------------------------------------------------ epilogue (warps 0-15)
        const int quad = warp & 3;        // TMEM lane quadrant this warp may access
        const int cg = warp >> 2;         // which 32 columns (tokens)
        const int row = quad * 32 + lane;  // weight row within the tile
        const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(cg * 32);
        float acc[32];  // running sums of this thread's 32 tokens
#pragma unroll
        for (int j = 0; j < 32; j++) acc[j] = 0.0f;
        // running state instead of per-block index arithmetic: the accumulator columns of
        // block b (S_BUFS of them in turn), its scale slot (SC_SLOTS in turn) and the
        // mma_done barrier of block b (DONE_RING in turn, phase b / DONE_RING)
        uint32_t s_cols = lane_base;
        int sbi = 0, sci = 0, dri = 0;
        uint32_t d_parity = 0;
        const float* scw_row = scw + row;
        const float* scx_cg = scx + cg * 32;
        const float* scm_row = scm + row;
        const float* scs_cg = scs + cg * 32;
        for (int b = 0; b < nb; b++) {  // blocks in order
            // warp-uniform: the TMEM loads below are warp-collective
            if (!__all_sync(0xffffffffu, wait_or_abort(bars.mma_done(dri), d_parity, abort_flag))) break;
            tc_fence_after();
            const int so = sci * BN;  // scale slot offset (BM == BN)
            const uint32_t dwb = __float_as_uint(scw_row[so]);
            const uint64_t dw2 = f2_pack(dwb, dwb);
            const uint4* dxs = reinterpret_cast<const uint4*>(scx_cg + so);
            // min formats: y += m_w * (d_x * sum(a)) after the block's value term
            const float mw = L::HAS_MIN ? scm_row[so] : 0.0f;
            const uint4* css = reinterpret_cast<const uint4*>(scs_cg + so);
            // the block's 32 sums in quarters of 8 columns: each quarter's TMEM load is
            // issued before the previous quarter is folded, so the load of one overlaps
            // the arithmetic of the other (a wait covers every load issued before it)
            uint32_t v[2][8];
            tmem_ld8(s_cols, v[0]);
            tmem_ld_wait_regs8(v[0]);
#pragma unroll
            for (int q = 0; q < 4; q++) {
                if (q < 3) tmem_ld8(s_cols + (uint32_t)(8 * (q + 1)), v[(q + 1) & 1]);
                const uint32_t* u = v[q & 1];
#pragma unroll
                for (int i = 0; i < 2; i++) {  // tokens t = 8q + 4i .. 8q + 4i + 3
                    // the scale products d_w*d_x[t] two at a time (the d_x pairs arrive as aligned
                    // register pairs), then one scalar FMA per sum reading the product's halves:
                    // no register-pair assembly of the loaded sums
                    const uint4 dx4 = dxs[2 * q + i];
                    const uint64_t sc0 = f2_mul(dw2, f2_pack(dx4.x, dx4.y));
                    const uint64_t sc1 = f2_mul(dw2, f2_pack(dx4.z, dx4.w));
                    const int t = 8 * q + 4 * i;
                    acc[t] = fmaf(__uint_as_float(u[4 * i]), __uint_as_float((uint32_t)sc0), acc[t]);
                    acc[t + 1] = fmaf(__uint_as_float(u[4 * i + 1]), __uint_as_float((uint32_t)(sc0 >> 32)), acc[t + 1]);
                    acc[t + 2] = fmaf(__uint_as_float(u[4 * i + 2]), __uint_as_float((uint32_t)sc1), acc[t + 2]);
                    acc[t + 3] = fmaf(__uint_as_float(u[4 * i + 3]), __uint_as_float((uint32_t)(sc1 >> 32)), acc[t + 3]);
                    if (L::HAS_MIN) {
                        const uint4 cs4 = css[2 * q + i];
                        acc[t] = fmaf(mw, __uint_as_float(cs4.x), acc[t]);
                        acc[t + 1] = fmaf(mw, __uint_as_float(cs4.y), acc[t + 1]);
                        acc[t + 2] = fmaf(mw, __uint_as_float(cs4.z), acc[t + 2]);
                        acc[t + 3] = fmaf(mw, __uint_as_float(cs4.w), acc[t + 3]);
                    }
                }
                if (q < 3) tmem_ld_wait_regs8(v[(q + 1) & 1]);
                if (q == 2) {  // all four quarters are in registers: the accumulator may be reused
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bars.acc_empty(sbi));
                }
            }
            if (++sbi == S_BUFS) {
                sbi = 0;
                s_cols = lane_base;
            } else {
                s_cols += BN;
            }
            sci = (sci + 1) & (SC_SLOTS - 1);
            if (++dri == DONE_RING) {
                dri = 0;
                d_parity ^= 1u;
            }
        }
        if (pdl) pdl_wait();  // Y may be read or written by the previous kernel
        const int o = o0 + row;
        if (!*abort_flag && o < N) {
#pragma unroll
            for (int j = 0; j < 32; j++) {
                const int t = t0 + cg * 32 + j;
                if (t < M && QMM_IN_BOUNDS(g_matmul_error, (size_t)t * N + o, (size_t)M * N))
                    Y[(size_t)t * N + o] = acc[j];
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == TMA_WARP) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
    }
}

}  // namespace mm

// ------------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

bool make_row_map(CUtensorMap* map, const void* base, uint64_t row_bytes, uint64_t rows, uint32_t box_bytes,
                  int elem_bytes) {
    EncodeTiledFn fn = encode_fn();
    if (!fn || (elem_bytes != 2 && elem_bytes != 8) || row_bytes % elem_bytes || box_bytes % 16) return false;
    const cuuint64_t dims[2] = {row_bytes / elem_bytes, rows};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_bytes / (uint32_t)elem_bytes, 128};
    const cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType t = elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT64;
    return fn(map, t, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The tensor-core path needs 16-byte row strides (K a multiple of 256) and
// enough tokens to fill a tile reasonably; other shapes run one matvec per token.
static bool tensor_core_shape(int64_t M, int64_t K) { return K % 256 == 0 && M >= 8; }

// One launch of the tensor-core kernel; XP: the activation operands were prepared
// into xp by q8_0_xprep_kernel (xq is then not read).
template <int WT, bool XP>
static qmm_status matmul_q_kernel_launch(const void* W, const void* xq, const uint8_t* xp, float* Y, int64_t M,
                                         int64_t N, int64_t K, cudaStream_t stream, bool pdl) {
    using L = mm::Lay<WT, XP>;
    CUtensorMap wmap, xmap;
    if (!make_row_map(&wmap, W, row_bytes_of(WT, K), (uint64_t)N, mm::KB * L::WB, 2)) return QMM_E_CUDA;
    if (XP) {
        xmap = CUtensorMap{};  // not read
    } else if (!make_row_map(&xmap, xq, row_bytes_of(QMM_Q8_0, K), (uint64_t)M, mm::KB * 34, 2)) {
        return QMM_E_CUDA;
    }
    static PerDeviceOnce attr_once;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return QMM_E_CUDA;
    const qmm_status ast = attr_once.run(dev, [] {
        return cudaFuncSetAttribute(mm::matmul_q_kernel<WT, XP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    L::SMEM_BYTES) == cudaSuccess
                   ? QMM_OK
                   : QMM_E_CUDA;
    });
    if (ast != QMM_OK) return ast;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((N + mm::BM - 1) / mm::BM), (unsigned)((M + mm::BN - 1) / mm::BN));
    cfg.blockDim = dim3(mm::Roles<XP>::THREADS);
    cfg.dynamicSmemBytes = L::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    const cudaError_t e =
        cudaLaunchKernelEx(&cfg, mm::matmul_q_kernel<WT, XP>, wmap, xmap, xp, Y, (int)M, (int)N, (int)K, pdl ? 1 : 0);
    return e == cudaSuccess ? QMM_OK : QMM_E_CUDA;
}

// Q4_1 and Q5_1 convert the activation once, in a pre-pass, into a stream-ordered
// workspace (cudaMallocAsync / cudaFreeAsync on the caller's stream: ~4.5 MB for
// 512 tokens at K = 4096): 10-11% faster at M = 128, 512 and 2048, their
// in-kernel conversion also summing every block's codes for the min term.  For
// Q4_0, Q8_0 and Q5_0 the pre-pass measured 4-7% slower, and without a workspace
// (no pool memory, or inside qmm_linear_noalloc) every CTA converts it too.
template <int WT>
static qmm_status matmul_q_launch(const void* W, const void* xq, float* Y, int64_t M, int64_t N, int64_t K,
                                  cudaStream_t stream, bool pdl) {
    if (!tensor_core_shape(M, K)) {
        const size_t xrb = row_bytes_of(QMM_Q8_0, K);
        for (int64_t t = 0; t < M; t++) {
            qmm_status st = matvec_dispatch(WT, W, (const uint8_t*)xq + t * xrb, Y + t * N, N, K, stream, pdl);
            if (st != QMM_OK) return st;
        }
        return QMM_OK;
    }
    if ((N + mm::BM - 1) / mm::BM > 0x7FFFFFFF || (M + mm::BN - 1) / mm::BN > 65535) return QMM_E_SHAPE;
    if (mm::Lay<WT>::HAS_MIN && !tl_no_workspace_alloc) {
        using LX = mm::Lay<WT, true>;
        const int64_t ntt = (M + mm::BN - 1) / mm::BN, nchunks = K / 32 / mm::KB;
        const size_t bytes = (size_t)(ntt * nchunks) * LX::XPS;
        void* buf = nullptr;
        if (cudaMallocAsync(&buf, bytes, stream) == cudaSuccess) {
            uint8_t* xp = static_cast<uint8_t*>(buf);
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3((unsigned)(nchunks * mm::KB), (unsigned)ntt);
            cfg.blockDim = dim3(mm::BN);
            cfg.stream = stream;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[0].val.programmaticStreamSerializationAllowed = 1;
            cfg.attrs = attr;
            cfg.numAttrs = pdl ? 1 : 0;
            const cudaError_t e =
                LX::HAS_MIN ? cudaLaunchKernelEx(&cfg, mm::q8_0_xprep_kernel<true>, (const uint8_t*)xq, xp, (int)M,
                                                 (int)nchunks, (int)LX::XPS, pdl ? 1 : 0)
                            : cudaLaunchKernelEx(&cfg, mm::q8_0_xprep_kernel<false>, (const uint8_t*)xq, xp, (int)M,
                                                 (int)nchunks, (int)LX::XPS, pdl ? 1 : 0);
            qmm_status st = e == cudaSuccess ? QMM_OK : QMM_E_CUDA;
            if (st == QMM_OK) st = matmul_q_kernel_launch<WT, true>(W, xq, xp, Y, M, N, K, stream, true);
            if (cudaFreeAsync(buf, stream) != cudaSuccess && st == QMM_OK) st = QMM_E_CUDA;
            return st;
        }
        (void)cudaGetLastError();  // no workspace: convert in the kernel
    }
    return matmul_q_kernel_launch<WT, false>(W, xq, nullptr, Y, M, N, K, stream, pdl);
}

// Whether an M-token multiply of this weight type takes a tensor-core prefill
// kernel (after one quantization of all M rows) rather than a launch per token.
// Q4_0 takes it for every M > 1 (its launcher runs per-token matvecs itself on
// shapes the tiles do not take); the other 32-value formats only on shapes the
// tiles take.
bool prefill_on_tensor_cores(int wt, int64_t M, int64_t K) {
    if (wt == QMM_Q4_0) return M > 1;
    if (wt == QMM_Q8_0 || wt == QMM_Q4_1 || wt == QMM_Q5_0 || wt == QMM_Q5_1) return M > 1 && tensor_core_shape(M, K);
    return kq_uses_tensor_cores(wt, M, K);
}

qmm_status prefill_launch(int wt, const void* W, const void* xq, float* Y, int64_t M, int64_t N, int64_t K,
                          cudaStream_t stream, bool pdl) {
    switch (wt) {
    case QMM_Q4_0: return matmul_q_launch<QMM_Q4_0>(W, xq, Y, M, N, K, stream, pdl);
    case QMM_Q8_0: return matmul_q_launch<QMM_Q8_0>(W, xq, Y, M, N, K, stream, pdl);
    case QMM_Q4_1: return matmul_q_launch<QMM_Q4_1>(W, xq, Y, M, N, K, stream, pdl);
    case QMM_Q5_0: return matmul_q_launch<QMM_Q5_0>(W, xq, Y, M, N, K, stream, pdl);
    case QMM_Q5_1: return matmul_q_launch<QMM_Q5_1>(W, xq, Y, M, N, K, stream, pdl);
    default: return matmul_kq_launch(wt, W, xq, Y, M, N, K, stream, pdl);
    }
}

}  // namespace qmm

using namespace qmm;

extern "C" {


static qmm_status matmul_public(int wt, const void* W, const void* xq, float* Y, int64_t M, int64_t N, int64_t K,
                                qmm_stream_t stream) {
    if (!W || !xq || !Y) return QMM_E_NULL;
    qmm_status st = check_shape(wt, M, N, K);
    if (st != QMM_OK) return st;
    if (!aligned16(W) || !aligned16(xq) || !aligned16(Y)) return QMM_E_ALIGN;
    return prefill_launch(wt, W, xq, Y, M, N, K, (cudaStream_t)stream, true);
}

qmm_status qmm_matmul_q4_0(const void* W, const void* xq, float* Y, int64_t M, int64_t N, int64_t K,
                           qmm_stream_t stream) {
    return matmul_public(QMM_Q4_0, W, xq, Y, M, N, K, stream);
}
qmm_status qmm_matmul_q8_0(const void* W, const void* xq, float* Y, int64_t M, int64_t N, int64_t K,
                           qmm_stream_t stream) {
    return matmul_public(QMM_Q8_0, W, xq, Y, M, N, K, stream);
}
qmm_status qmm_matmul_q4_1(const void* W, const void* xq, float* Y, int64_t M, int64_t N, int64_t K,
                           qmm_stream_t stream) {
    return matmul_public(QMM_Q4_1, W, xq, Y, M, N, K, stream);
}
qmm_status qmm_matmul_q5_0(const void* W, const void* xq, float* Y, int64_t M, int64_t N, int64_t K,
                           qmm_stream_t stream) {
    return matmul_public(QMM_Q5_0, W, xq, Y, M, N, K, stream);
}
qmm_status qmm_matmul_q5_1(const void* W, const void* xq, float* Y, int64_t M, int64_t N, int64_t K,
                           qmm_stream_t stream) {
    return matmul_public(QMM_Q5_1, W, xq, Y, M, N, K, stream);
}

unsigned qmm_internal_matmul_error(int clear) {
    unsigned v = 0;
    cudaMemcpyFromSymbol(&v, g_matmul_error, sizeof(v));
    if (clear) {
        const unsigned z = 0;
        cudaMemcpyToSymbol(g_matmul_error, &z, sizeof(z));
    }
    return v;
}

}  // extern "C"
