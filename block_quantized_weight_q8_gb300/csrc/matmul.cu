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
// One CTA per output tile of 128 weight rows x 128 tokens, 28 warps:
//   warp 0   producer: 2-D TMA loads of the raw weight bytes (128 rows x 8 blocks)
//            and the raw activation bytes (128 tokens x 8 blocks) into a ring of
//            raw stages; also owns the tensor-memory allocation
//   warp 1   MMA issuer: per pair of blocks, two tcgen05.mma (K = 16 each) per
//            block into its own 128-column TMEM accumulator, then one
//            tcgen05.commit for the pair
//   warps 2-4, 6-8, 10-11  converters (four for weight rows, four for tokens):
//            each thread loads its row of the raw stage into registers with
//            16-byte loads, then writes each block as fp16 operands in the UMMA
//            K-major core-matrix layout (8 rows x 16 bytes per core matrix) plus
//            its f32 scale; warps 5 and 9 stay idle so that the MMA issuer's
//            scheduler carries no converter work
//   warps 12-27 epilogue: tcgen05.ld of each block's exact sums (32 tokens of one
//            weight row per thread), y += v * (d_w*d_x) in registers in block
//            order, then the token-major store
// Blocks move between the roles in pairs (one barrier handshake per two blocks);
// all waits are bounded; a timeout records QMM_E_TIMEOUT, every warp still
// reaches the end, and TMEM is freed.
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
constexpr int ACC_PAIRS = 2;       // accumulator pairs: two blocks' sums per handshake (4 x 128 columns)
constexpr int X_RAW = BN * KB * 34;   // 34816
constexpr int OP_A = BM * 32 * 2;     // 8192: fp16 weights of one block
constexpr int OP_B = BN * 32 * 2;     // 8192: fp16 activations of one block
constexpr int NUM_CONV_WARPS = 8, NUM_EPI_WARPS = 16;  // converters: 4 for weights, 4 for activations
// Warps 0-11: producer (0), MMA issuer (1), converters (2-4, 6-8, 10-11), two
// idle warps (5, 9) that keep the MMA issuer's scheduler free of converter work;
// warps 12-27: epilogue (warp % 4 is the TMEM lane quadrant it may read).
constexpr int EPI0 = 12;
constexpr int THREADS = (EPI0 + NUM_EPI_WARPS) * 32;  // 896
constexpr int TMEM_COLS = 2 * ACC_PAIRS * BN;  // 512: four 128-column accumulators

__device__ __forceinline__ int converter_index(int warp) {  // 0..7, or -1 for other warps
    return (warp >= 2 && warp < EPI0 && warp != 5 && warp != 9) ? warp - 2 - (warp > 5) - (warp > 9) : -1;
}

// Weight block bytes of the 32-value formats (Q4_0 18, Q8_0 34, Q4_1 20, Q5_0 22, Q5_1 24).
__host__ __device__ constexpr int block_bytes32(int wt) {
    return wt == QMM_Q8_0 ? 34 : wt == QMM_Q4_1 ? 20 : wt == QMM_Q5_0 ? 22 : wt == QMM_Q5_1 ? 24 : 18;
}

// Shared memory layout per weight format (offsets from the 1024-byte aligned
// dynamic shared memory base).  Q4_0 keeps 32 scale slots; the larger raw stages
// of the other formats leave room for 16.  (A third operand pair for Q4_0, in
// place of 16 scale slots, measured no faster.)  Q4_1 and Q5_1 also carry each
// row's m_w and each token's d_x * sum(a) per block, for the min term.
template <int WT>
struct Lay {
    static constexpr int WB = block_bytes32(WT);
    static constexpr bool HAS_MIN = WT == QMM_Q4_1 || WT == QMM_Q5_1;
    static constexpr int PAIRS = 2;                             // operand pair slots (converted blocks in flight / 2)
    static constexpr int OPS = 2 * PAIRS;
    static constexpr int SC_SLOTS = WT == QMM_Q4_0 ? 32 : 16;  // block scales in flight (outlive the operands)
    static constexpr int SCP = SC_SLOTS / 2;                   // ... in pairs
    static constexpr int W_RAW = BM * KB * WB;
    static constexpr int RAW_BYTES = W_RAW + X_RAW;
    static constexpr int OFF_RAW = 0;
    static constexpr int OFF_OPA = OFF_RAW + RAW_STAGES * RAW_BYTES;
    static constexpr int OFF_OPB = OFF_OPA + OPS * OP_A;
    static constexpr int OFF_SCW = OFF_OPB + OPS * OP_B;
    static constexpr int OFF_SCX = OFF_SCW + SC_SLOTS * BM * 4;
    static constexpr int OFF_SCM = OFF_SCX + SC_SLOTS * BN * 4;            // m_w per row (min formats)
    static constexpr int OFF_SCS = OFF_SCM + (HAS_MIN ? SC_SLOTS * BM * 4 : 0);  // d_x * sum(a) per token
    static constexpr int OFF_BAR = OFF_SCS + (HAS_MIN ? SC_SLOTS * BN * 4 : 0);
    // barriers: raw_full[2] raw_empty[2] op_full[PAIRS] op_empty[PAIRS] acc_full[2] acc_empty[2] sc_empty[SCP]
    static constexpr int NBARS = 2 * RAW_STAGES + 2 * PAIRS + 2 * ACC_PAIRS + SCP;
    static constexpr int OFF_TMEM = OFF_BAR + NBARS * 8;
    static constexpr int SMEM_BYTES = OFF_TMEM + 16;
};
static_assert(Lay<QMM_Q4_0>::SMEM_BYTES <= 232448 && Lay<QMM_Q8_0>::SMEM_BYTES <= 232448 &&
                  Lay<QMM_Q4_1>::SMEM_BYTES <= 232448 && Lay<QMM_Q5_0>::SMEM_BYTES <= 232448 &&
                  Lay<QMM_Q5_1>::SMEM_BYTES <= 232448,
              "prefill smem");
static_assert(KB % 4 == 0, "pairs must not straddle the activation converter's 4-block windows");

struct Bars {
    uint32_t base;
    int pairs;  // operand pair slots
    __device__ uint32_t raw_full(int i) const { return base + 8u * i; }
    __device__ uint32_t raw_empty(int i) const { return base + 8u * (RAW_STAGES + i); }
    // operand pair slot i: written by the converters / read by the tensor core (one tcgen05.commit)
    __device__ uint32_t op_full(int i) const { return base + 8u * (2 * RAW_STAGES + i); }
    __device__ uint32_t op_empty(int i) const { return base + 8u * (2 * RAW_STAGES + pairs + i); }
    // accumulator pair i: both blocks' sums complete (one tcgen05.commit) / read into registers
    __device__ uint32_t acc_full(int i) const { return base + 8u * (2 * RAW_STAGES + 2 * pairs + i); }
    __device__ uint32_t acc_empty(int i) const { return base + 8u * (2 * RAW_STAGES + 2 * pairs + ACC_PAIRS + i); }
    // scale pair slot i read by the epilogue
    __device__ uint32_t sc_empty(int i) const {
        return base + 8u * (2 * RAW_STAGES + 2 * pairs + 2 * ACC_PAIRS + i);
    }
};

// wait with a time limit; on failure set the error word and the CTA's abort flag.
// The fast path (phase already complete) is a single try_wait: the roles here
// share their schedulers with FP32-heavy warps, so every instruction counts.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (mbar_wait_bounded(bar, parity, kWaitLimitNs)) return true;
    atomicOr(&g_matmul_error, kErrTimeout);
    *abort_flag = 1;
    return false;
}

template <int WT>
__global__ void __launch_bounds__(THREADS, 1)
    matmul_q_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap xmap,
                    float* __restrict__ Y, int M, int N, int K, int pdl) {
    if (pdl) pdl_launch_dependents();
    // used directly (not re-aligned by integer arithmetic) so that the compiler
    // keeps every access in the shared state space
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sbase = smem_u32(smem);
    if (sbase & 127u) {  // the TMA destinations and operand tiles need 128-byte alignment
        if (threadIdx.x == 0) atomicOr(&g_matmul_error, kErrTimeout);
        return;
    }
    using L = Lay<WT>;
    if (!QMM_IN_BOUNDS(g_matmul_error, L::SMEM_BYTES - 1, dynamic_smem_bytes())) return;  // the layout must fit
    constexpr int SC_SLOTS = L::SC_SLOTS, SCP = L::SCP, W_RAW = L::W_RAW, RAW_BYTES = L::RAW_BYTES, WB = L::WB,
                  PAIRS = L::PAIRS;
    const Bars bars{sbase + L::OFF_BAR, PAIRS};
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
            mbar_init(bars.raw_empty(i), NUM_CONV_WARPS);
        }
        for (int i = 0; i < PAIRS; i++) {
            mbar_init(bars.op_full(i), NUM_CONV_WARPS);
            mbar_init(bars.op_empty(i), 1);
        }
        for (int i = 0; i < ACC_PAIRS; i++) {
            mbar_init(bars.acc_full(i), 1);
            mbar_init(bars.acc_empty(i), NUM_EPI_WARPS);
        }
        for (int i = 0; i < SCP; i++) mbar_init(bars.sc_empty(i), NUM_EPI_WARPS);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {  // allocate the TMEM accumulators (whole warp)
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int cw = converter_index(warp);

    if (warp == 0) {
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
                tma_load_2d(dst + W_RAW, &xmap, c * (KB * 34 / 2), t0, bars.raw_full(s));
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = instr_desc_f16(BM, BN);
            // descriptors of slot 0; slot os adds os * OP_A (>> 4) to the address field
            const uint64_t a0 = smem_desc(sbase + L::OFF_OPA, 128, 512);
            const uint64_t b0 = smem_desc(sbase + L::OFF_OPB, 128, 512);
            for (int p = 0; p < nb / 2; p++) {  // blocks 2p and 2p+1 per handshake
                const int ps = p % PAIRS, ap = p % ACC_PAIRS;
                if (!wait_or_abort(bars.op_full(ps), (p / PAIRS) & 1, abort_flag)) break;
                if (p >= ACC_PAIRS && !wait_or_abort(bars.acc_empty(ap), ((p / ACC_PAIRS) - 1) & 1, abort_flag))
                    break;
                tc_fence_after();
#pragma unroll
                for (int i = 0; i < 2; i++) {
                    const int os = 2 * ps + i;
                    const uint64_t ad = a0 + (uint64_t)(os * (OP_A >> 4));
                    const uint64_t bd = b0 + (uint64_t)(os * (OP_B >> 4));
                    const uint32_t d = tmem + (uint32_t)((2 * ap + i) * BN);
                    mma_f16(d, ad, bd, idesc, 0);                            // K 0..15: core matrices 0, 1
                    mma_f16(d, ad + (256 >> 4), bd + (256 >> 4), idesc, 1);  // K 16..31: core matrices 2, 3
                }
                mma_commit(bars.op_empty(ps));
                mma_commit(bars.acc_full(ap));
            }
        }
    } else if (cw >= 0) {
        // ------------------------------------------------------------ converters
        // Blocks go in pairs: the slots of pair p are taken (operands freed by the
        // MMAs of pair p - PAIRS, scales by the epilogue of pair p - SCP) before
        // its first block, and handed to the MMA issuer after its second.
        const bool is_w = cw < NUM_CONV_WARPS / 2;
        const int r = (cw % (NUM_CONV_WARPS / 2)) * 32 + lane;  // weight row or token, 0..127
        for (int c = 0; c < nchunks; c++) {
            const int s = c % RAW_STAGES;
            if (!wait_or_abort(bars.raw_full(s), (c / RAW_STAGES) & 1, abort_flag)) break;
            if (WT == QMM_Q4_0 && is_w) {
                // this Q4_0 weight row's 8 blocks: 144 bytes, 16-byte aligned
                uint32_t raw[36];
                const uint4* src = reinterpret_cast<const uint4*>(smem + L::OFF_RAW + s * RAW_BYTES + r * (KB * 18));
#pragma unroll
                for (int i = 0; i < 9; i++) {
                    const uint4 v = src[i];
                    raw[4 * i] = v.x; raw[4 * i + 1] = v.y; raw[4 * i + 2] = v.z; raw[4 * i + 3] = v.w;
                }
#pragma unroll
                for (int lb = 0; lb < KB; lb++) {
                    const int b = c * KB + lb, p = b >> 1, ps = p % PAIRS, os = 2 * ps + (b & 1), ss = b % SC_SLOTS;
                    if ((b & 1) == 0) {
                        if (p >= PAIRS && !wait_or_abort(bars.op_empty(ps), ((p / PAIRS) - 1) & 1, abort_flag)) break;
                        if (p >= SCP && !wait_or_abort(bars.sc_empty(p % SCP), ((p / SCP) - 1) & 1, abort_flag))
                            break;
                    }
                    // block lb: f16 d at byte 18*lb, nibbles at 18*lb + 2 (element j low, j+16 high)
                    const int off = 18 * lb;
                    const uint32_t dbits = __funnelshift_r(raw[off / 4], raw[off / 4 + 1], 8 * (off % 4)) & 0xFFFFu;
                    uint32_t lo[4], hi[4];
#pragma unroll
                    for (int i = 0; i < 4; i++) {
                        const int qo = off + 2 + 4 * i;
                        const uint32_t q = __funnelshift_r(raw[qo / 4], raw[qo / 4 + 1], 8 * (qo % 4));
                        lo[i] = q & 0x0F0F0F0Fu;
                        hi[i] = (q >> 4) & 0x0F0F0F0Fu;
                    }
                    const uint32_t m8 = 0x64086408u;  // (1032, 1032): 1024 + n - 1032 = n - 8
                    uint8_t* A = smem + L::OFF_OPA + os * OP_A;
#pragma unroll
                    for (int kq = 0; kq < 4; kq++) {  // elements 8kq..8kq+7
                        const uint32_t w0 = kq < 2 ? lo[2 * kq] : hi[2 * (kq - 2)];
                        const uint32_t w1 = kq < 2 ? lo[2 * kq + 1] : hi[2 * (kq - 2) + 1];
                        uint4 v;
                        v.x = h2_sub(bytes_to_h2(w0, 0x5140), m8);
                        v.y = h2_sub(bytes_to_h2(w0, 0x7362), m8);
                        v.z = h2_sub(bytes_to_h2(w1, 0x5140), m8);
                        v.w = h2_sub(bytes_to_h2(w1, 0x7362), m8);
                        *reinterpret_cast<uint4*>(A + op_off(r, kq)) = v;
                    }
                    reinterpret_cast<float*>(smem + L::OFF_SCW)[ss * BM + r] = h2f(dbits);
                    if (b & 1) {
                        fence_proxy_async_smem();  // the operands are read by the tensor core (async proxy)
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bars.op_full(ps));
                    }
                }
            } else if (is_w && (WT == QMM_Q4_1 || WT == QMM_Q5_0 || WT == QMM_Q5_1)) {
                // this weight row's 8 blocks (160, 176 or 192 bytes, 16-byte aligned), read as two
                // windows of 4 blocks starting at the 16-byte boundary at or below each window's
                // first byte.  Q4_1: d, m, qs@4; Q5_0: d, qh@2, qs@6; Q5_1: d, m, qh@4, qs@8;
                // element j is the low nibble of qs[j], element j+16 the high one, and bit e of
                // qh is element e's fifth bit.
                constexpr int OFF_Q = WT == QMM_Q4_1 ? 4 : WT == QMM_Q5_0 ? 6 : 8;
                constexpr int OFF_H = WT == QMM_Q5_0 ? 2 : 4;
                constexpr bool FIVE = WT != QMM_Q4_1;
                // fp16 bits of (1024 + byte) minus 1024 (codes 0..31) or 1040 (Q5_0: code - 16)
                constexpr uint32_t magic = WT == QMM_Q5_0 ? 0x64106410u : 0x64006400u;
                const uint8_t* rowp = smem + L::OFF_RAW + s * RAW_BYTES + r * (KB * WB);
#pragma unroll
                for (int h = 0; h < 2; h++) {
                    const int start = 4 * WB * h, base16 = start & ~15, off0 = start - base16;
                    const int nv = (off0 + 4 * WB + 15) / 16;  // 16-byte loads: 5 or 6
                    uint32_t raw[25];
                    raw[24] = 0;
                    const uint4* src = reinterpret_cast<const uint4*>(rowp + base16);
#pragma unroll
                    for (int i = 0; i < 6; i++) {
                        if (i < nv) {
                            const uint4 v = src[i];
                            raw[4 * i] = v.x; raw[4 * i + 1] = v.y; raw[4 * i + 2] = v.z; raw[4 * i + 3] = v.w;
                        } else {
                            raw[4 * i] = raw[4 * i + 1] = raw[4 * i + 2] = raw[4 * i + 3] = 0;
                        }
                    }
#pragma unroll
                    for (int lq = 0; lq < KB / 2; lq++) {
                        const int lb = 4 * h + lq;
                        const int b = c * KB + lb, p = b >> 1, ps = p % PAIRS, os = 2 * ps + (b & 1),
                                  ss = b % SC_SLOTS;
                        if ((b & 1) == 0) {
                            if (p >= PAIRS &&
                                !wait_or_abort(bars.op_empty(ps), ((p / PAIRS) - 1) & 1, abort_flag))
                                break;
                            if (p >= SCP && !wait_or_abort(bars.sc_empty(p % SCP), ((p / SCP) - 1) & 1, abort_flag))
                                break;
                        }
                        const int off = off0 + WB * lq;  // the block's first byte in the window
                        auto word_at = [&](int o) -> uint32_t {
                            return (o % 4 == 0) ? raw[o / 4] : __funnelshift_r(raw[o / 4], raw[o / 4 + 1], 8 * (o % 4));
                        };
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
                        uint8_t* A = smem + L::OFF_OPA + os * OP_A;
#pragma unroll
                        for (int kq = 0; kq < 4; kq++) {  // elements 8kq..8kq+7
                            const uint32_t w0 = kq < 2 ? lo[2 * kq] : hi[2 * (kq - 2)];
                            const uint32_t w1 = kq < 2 ? lo[2 * kq + 1] : hi[2 * (kq - 2) + 1];
                            uint4 v;
                            v.x = h2_sub(bytes_to_h2(w0, 0x5140), magic);
                            v.y = h2_sub(bytes_to_h2(w0, 0x7362), magic);
                            v.z = h2_sub(bytes_to_h2(w1, 0x5140), magic);
                            v.w = h2_sub(bytes_to_h2(w1, 0x7362), magic);
                            *reinterpret_cast<uint4*>(A + op_off(r, kq)) = v;
                        }
                        reinterpret_cast<float*>(smem + L::OFF_SCW)[ss * BM + r] = h2f(dm & 0xFFFFu);
                        if (L::HAS_MIN) reinterpret_cast<float*>(smem + L::OFF_SCM)[ss * BM + r] = h2f(dm >> 16);
                        if (b & 1) {
                            fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(bars.op_full(ps));
                        }
                    }
                }
            } else {
                // this token's (or Q8_0 weight row's) 8 blocks: 272 bytes, 16-byte aligned,
                // read as two windows of 144 bytes (bytes 0..143 hold blocks 0-3, bytes
                // 128..271 hold blocks 4-7)
                const uint8_t* row = smem + L::OFF_RAW + s * RAW_BYTES + (is_w ? 0 : W_RAW) + r * (KB * 34);
                uint8_t* const opbase = smem + (is_w ? L::OFF_OPA : L::OFF_OPB);
                float* const scbase = reinterpret_cast<float*>(smem + (is_w ? L::OFF_SCW : L::OFF_SCX));
#pragma unroll
                for (int h = 0; h < 2; h++) {
                    uint32_t raw[36];
                    const uint4* src = reinterpret_cast<const uint4*>(row + 128 * h);
#pragma unroll
                    for (int i = 0; i < 9; i++) {
                        const uint4 v = src[i];
                        raw[4 * i] = v.x; raw[4 * i + 1] = v.y; raw[4 * i + 2] = v.z; raw[4 * i + 3] = v.w;
                    }
#pragma unroll
                    for (int lq = 0; lq < KB / 2; lq++) {
                        const int lb = 4 * h + lq;
                        const int b = c * KB + lb, p = b >> 1, ps = p % PAIRS, os = 2 * ps + (b & 1),
                                  ss = b % SC_SLOTS;
                        if ((b & 1) == 0) {
                            if (p >= PAIRS &&
                                !wait_or_abort(bars.op_empty(ps), ((p / PAIRS) - 1) & 1, abort_flag))
                                break;
                            if (p >= SCP && !wait_or_abort(bars.sc_empty(p % SCP), ((p / SCP) - 1) & 1, abort_flag))
                                break;
                        }
                        // block lb: f16 d at byte 34*lb, 32 int8 codes at 34*lb + 2 (window-relative)
                        const int off = 34 * lb - 128 * h;
                        const uint32_t dbits =
                            __funnelshift_r(raw[off / 4], raw[off / 4 + 1], 8 * (off % 4)) & 0xFFFFu;
                        const uint32_t m128 = 0x64806480u;  // (1152, 1152): 1024 + (a + 128) - 1152 = a
                        static_assert(OP_A == OP_B && BM == BN, "one converter for both operands");
                        uint8_t* Bop = opbase + os * OP_B;
                        int asum = 0;  // sum of the block's codes (min formats: the token's m_w term)
#pragma unroll
                        for (int kq = 0; kq < 4; kq++) {  // elements 8kq..8kq+7: code words 2kq, 2kq+1
                            const int q0 = off + 2 + 8 * kq, q1 = q0 + 4;
                            const uint32_t c0 = __funnelshift_r(raw[q0 / 4], raw[q0 / 4 + 1], 8 * (q0 % 4));
                            const uint32_t c1 = __funnelshift_r(raw[q1 / 4], raw[q1 / 4 + 1], 8 * (q1 % 4));
                            if (L::HAS_MIN) asum = __dp4a((int)c1, 0x01010101, __dp4a((int)c0, 0x01010101, asum));
                            const uint32_t w0 = c0 ^ 0x80808080u, w1 = c1 ^ 0x80808080u;
                            uint4 v;
                            v.x = h2_sub(bytes_to_h2(w0, 0x5140), m128);
                            v.y = h2_sub(bytes_to_h2(w0, 0x7362), m128);
                            v.z = h2_sub(bytes_to_h2(w1, 0x5140), m128);
                            v.w = h2_sub(bytes_to_h2(w1, 0x7362), m128);
                            *reinterpret_cast<uint4*>(Bop + op_off(r, kq)) = v;
                        }
                        scbase[ss * BN + r] = h2f(dbits);
                        if (L::HAS_MIN && !is_w)
                            reinterpret_cast<float*>(smem + L::OFF_SCS)[ss * BN + r] = h2f(dbits) * (float)asum;
                        if (b & 1) {
                            fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(bars.op_full(ps));
                        }
                    }
                }
            }
            // The raw stage goes back to the producer only once every value read from it
            // has been used: released right after the loads, the next chunk's TMA was seen
            // to overwrite a window whose loads the weight converter had just issued.
            __syncwarp();
            if (lane == 0) mbar_arrive(bars.raw_empty(s));
        }
    } else if (warp >= EPI0) {
        // ------------------------------------------------------------ epilogue
        const int e = warp - EPI0;        // 0..15
        const int quad = warp & 3;        // TMEM lane quadrant this warp may access
        const int cg = e >> 2;            // which 32 columns (tokens)
        const int row = quad * 32 + lane;  // weight row within the tile
        const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(cg * 32);
        uint64_t acc[16];  // running sums of tokens 2j, 2j+1 as packed f32 pairs
#pragma unroll
        for (int j = 0; j < 16; j++) acc[j] = 0;
        for (int p = 0; p < nb / 2; p++) {
            const int ap = p % ACC_PAIRS;
            if (!wait_or_abort(bars.acc_full(ap), (p / ACC_PAIRS) & 1, abort_flag)) break;
            tc_fence_after();
#pragma unroll 1
            for (int i = 0; i < 2; i++) {  // blocks 2p, 2p+1 in block order (not unrolled: registers)
                const int ss = (2 * p + i) % SC_SLOTS, ac = 2 * ap + i;
                const uint32_t dwb = __float_as_uint(scw[ss * BM + row]);
                const uint64_t dw2 = f2_pack(dwb, dwb);
                const uint64_t* dxs = reinterpret_cast<const uint64_t*>(scx + ss * BN + cg * 32);
                // min formats: y += m_w * (d_x * sum(a)) after the block's value term
                const uint32_t mwb = L::HAS_MIN ? __float_as_uint(scm[ss * BM + row]) : 0u;
                const uint64_t mw2 = f2_pack(mwb, mwb);
                const uint64_t* css = reinterpret_cast<const uint64_t*>(scs + ss * BN + cg * 32);
#pragma unroll
                for (int h = 0; h < 2; h++) {
                    uint32_t v[16];
                    tmem_ld16(lane_base + (uint32_t)(ac * BN + 16 * h), v);
                    tmem_ld_wait();
                    if (i == 1 && h == 1) {  // both blocks' sums are in registers: the accumulators may be reused
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bars.acc_empty(ap));
                    }
#pragma unroll
                    for (int j = 0; j < 8; j++) {
                        const uint64_t sc = f2_mul(dw2, dxs[8 * h + j]);  // (d_w*d_x[t], d_w*d_x[t+1])
                        acc[8 * h + j] = f2_fma(f2_pack(v[2 * j], v[2 * j + 1]), sc, acc[8 * h + j]);
                        if (L::HAS_MIN) acc[8 * h + j] = f2_fma(mw2, css[8 * h + j], acc[8 * h + j]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bars.sc_empty(p % SCP));
        }
        if (pdl) pdl_wait();  // Y may be read or written by the previous kernel
        const int o = o0 + row;
        if (!*abort_flag && o < N) {
#pragma unroll
            for (int j = 0; j < 32; j++) {
                const int t = t0 + cg * 32 + j;
                const uint32_t bits = (j & 1) ? (uint32_t)(acc[j >> 1] >> 32) : (uint32_t)acc[j >> 1];
                if (t < M && QMM_IN_BOUNDS(g_matmul_error, (size_t)t * N + o, (size_t)M * N))
                    Y[(size_t)t * N + o] = __uint_as_float(bits);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
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

// A 2-D map over `rows` rows of `row_bytes` bytes, viewed as 16-bit elements,
// with boxes of `box_bytes` x 128 rows; rows beyond the end read as zeros.
static bool make_map(CUtensorMap* map, const void* base, uint64_t row_bytes, uint64_t rows, uint32_t box_bytes) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {row_bytes / 2, rows};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_bytes / 2, 128};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The tensor-core path needs 16-byte row strides (K a multiple of 256) and
// enough tokens to fill a tile reasonably; other shapes run one matvec per token.
static bool tensor_core_shape(int64_t M, int64_t K) { return K % 256 == 0 && M >= 8; }

template <int WT>
static qmm_status matmul_q_launch(const void* W, const void* xq, float* Y, int64_t M, int64_t N, int64_t K,
                                  cudaStream_t stream, bool pdl) {
    using L = mm::Lay<WT>;
    if (!tensor_core_shape(M, K)) {
        const size_t xrb = row_bytes_of(QMM_Q8_0, K);
        for (int64_t t = 0; t < M; t++) {
            qmm_status st = matvec_dispatch(WT, W, (const uint8_t*)xq + t * xrb, Y + t * N, N, K, stream, pdl);
            if (st != QMM_OK) return st;
        }
        return QMM_OK;
    }
    if ((N + mm::BM - 1) / mm::BM > 0x7FFFFFFF || (M + mm::BN - 1) / mm::BN > 65535) return QMM_E_SHAPE;
    CUtensorMap wmap, xmap;
    if (!make_map(&wmap, W, row_bytes_of(WT, K), (uint64_t)N, mm::KB * L::WB) ||
        !make_map(&xmap, xq, row_bytes_of(QMM_Q8_0, K), (uint64_t)M, mm::KB * 34))
        return QMM_E_CUDA;
    static PerDeviceOnce attr_once;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return QMM_E_CUDA;
    const qmm_status ast = attr_once.run(dev, [] {
        return cudaFuncSetAttribute(mm::matmul_q_kernel<WT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    L::SMEM_BYTES) == cudaSuccess
                   ? QMM_OK
                   : QMM_E_CUDA;
    });
    if (ast != QMM_OK) return ast;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((N + mm::BM - 1) / mm::BM), (unsigned)((M + mm::BN - 1) / mm::BN));
    cfg.blockDim = dim3(mm::THREADS);
    cfg.dynamicSmemBytes = L::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    const cudaError_t e =
        cudaLaunchKernelEx(&cfg, mm::matmul_q_kernel<WT>, wmap, xmap, Y, (int)M, (int)N, (int)K, pdl ? 1 : 0);
    return e == cudaSuccess ? QMM_OK : QMM_E_CUDA;
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
