// pkv_prefill_tc.cu -- ragged paged prefill on the 5th-generation tensor cores
// (tcgen05, accumulators in tensor memory), bf16, head_dim 64 or 128; the same
// pipeline runs the group role of the shared-prefix decode (head_dim 128).
//
// Operation (AstrAI docs/guides/inference.md, "Attention Backend" prefill
// path; causal alignment from astrai/model/transformer.py
// process_attention_mask): entry b has q_len = qo_indptr[b+1] - qo_indptr[b]
// new tokens at the end of kv_len = kv_indptr[b+1] - kv_indptr[b] positions;
// packed query row qo_indptr[b] + i, head h attends to slots
// req_to_token[req_pool_indices[b], j] of kv head h / G for j <= P + i
// (P = kv_len - q_len) or j < kv_len when not causal.
//
// One CTA of 16 warps per (pair of query tiles, kv head, entry).  A query
// tile is 128 rows of (position, head-in-group) pairs; the CTA's two tiles A
// and B (rows [256 i, 256 i + 128) and the next 128) share every gathered
// K/V tile, which halves the gathered bytes per flop: a gather of random
// 256-byte rows beside the SM's own tensor, MUFU and TMEM traffic moves
// ~40 GB/s per SM, and with one 64 KB tile in flight that gather sets the
// tile period.  The warps specialise and hand work over through mbarriers
// (every wait bounded):
//  - producer warps 8..14 (224 threads): each 128-token K and V tile is
//    loaded with 16-byte loads (head_dim / 8 threads per token row, slot
//    indices staged in shared memory) into registers, then stored into a
//    2-slot ring once the tensor core has released the slot; tile 0 is
//    gathered while the other warps load the query tiles (the group role
//    copies with cp.async instead, see its producer);
//  - MMA warp 15 (one thread) issues, per tile j,
//      PV_A(j-1), S_A(j), PV_B(j-1), S_B(j)     (S = Q K^T, O += P V),
//    S as head_dim / 16 tcgen05.mma (M=128, N=128, K=16) and P.V as 8
//    (M=128, N=head_dim, K=16), so the tensor core works on one query tile
//    while the softmax runs on the other;
//  - softmax warps 0..7: warps w and w+4 share TMEM lanes 32(w%4).. and take
//    one 64-column half of each row.  A thread reads its 64 scores of S_X(j)
//    into registers once, exchanges its half's maximum with the other half
//    through shared memory and a named barrier, keeps a running
//    maximum that is only raised when the tile maximum exceeds it by more
//    than 2^8 (then its half of O_X is rescaled in TMEM -- P.V_X(j-1) is
//    complete, as it was issued before S_X(j)), and stores P = 2^(s - m) as
//    bf16 pairs over the S columns it has read; P.V reads P from TMEM as its
//    A operand.
// TMEM (512 columns): tile X in {A, B} has S (and P) at 256 X and O (head_dim
// columns) at 256 X + 128.  Q, K and V tiles use the 128-byte swizzle: a
// [rows x head_dim] bf16 tile is one or two 64-column halves of rows x 128 B,
// 16-byte chunk c of row r stored at chunk c ^ (r % 8), atoms 1024-byte
// aligned.
#include <atomic>

#include "pkv_common.cuh"
#include "pkv_launch.h"

namespace pkv {
namespace {

constexpr int kRows = 128;       // query rows per query tile (TMEM lanes)
constexpr int kTok = 128;        // kv tokens per tile
constexpr int kSoftmaxWarps = 8;
constexpr int kProducerWarps = 7;
constexpr int kMmaWarp = kSoftmaxWarps + kProducerWarps;
constexpr int kNT = (kMmaWarp + 1) * 32;                   // 512 threads
constexpr int kPT = kProducerWarps * 32;                   // 224 producer threads
// mbarriers
constexpr int kBarKFull = 0;     // [2 slots] count kPT: producer threads
constexpr int kBarKEmpty = 2;    // [2 slots] count 1: commit after the tile's S products
constexpr int kBarVFull = 4;     // [2 slots] count kPT
constexpr int kBarVEmpty = 6;    // [2 slots] count 1: commit after the tile's P.V products
constexpr int kBarSFull = 8;     // [2 query tiles] count 1: S_X(j) complete
constexpr int kBarPFull = 10;    // [2 query tiles] count 8: softmax warps have stored P_X(j)
constexpr int kBarODone = 12;    // [2 query tiles] count 1: the last P.V_X complete
constexpr int kNumBars = 14;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescale = 8.f;                            // lazy rescale threshold (log2 units)
static_assert(kGroupRows == 2 * kRows, "a group-role CTA holds two query tiles");
// group-role epilogue: each softmax warp stages 32 rows x 64 fp32 columns with
// a 16-byte row pad (conflict-free 16-byte stores) in the query + K tile area
constexpr int kStgPitch = 68;

// Shared-memory layout for head_dim D (64 or 128): Q, K and V tiles are
// [128 x D] bf16 (one or two 128-byte-swizzled 64-column halves).
template <int D>
struct TcLayout {
    static constexpr int kChunksRow = D / 8;                          // 16-byte chunks per row
    static constexpr int kChunks = (kTok * kChunksRow + kPT - 1) / kPT;   // per producer thread and tile
    static constexpr int kTileBytes = 128 * D * 2;                    // any [128 x D] bf16 tile
    static constexpr int kSmemQ = 0;                                  // [2] query tiles A, B
    static constexpr int kSmemK = 2 * kTileBytes;                     // [2] K slots
    static constexpr int kSmemV = kSmemK + 2 * kTileBytes;            // [2] V slots
    static constexpr int kSmemBar = kSmemV + 2 * kTileBytes;
    static constexpr int kSmemTmemAddr = kSmemBar + kNumBars * 8;
    static constexpr int kSmemAbort = kSmemTmemAddr + 4;
    static constexpr int kSmemRed = kSmemBar + 256;                   // [2 tiles][2 buffers][2 halves][kRows] float
    static constexpr int kSmemSlots = kSmemRed + 2 * 2 * 2 * kRows * 4;   // [2][kTok] int: producer's slot indices
    static constexpr int kSmemBytes = kSmemSlots + 2 * kTok * 4 + 1024;   // + alignment slack
    static_assert(D == 64 || D == 128, "head_dim 64 or 128");
    static_assert(kSmemAbort + 4 <= kSmemRed, "barrier area");
    static_assert(kSmemBytes <= 227 * 1024, "shared memory");
};
static_assert(kSoftmaxWarps * 32 * kStgPitch * 4 <= TcLayout<128>::kSmemV - TcLayout<128>::kSmemQ,
              "epilogue staging fits the Q and K tiles");

// byte offset of 16-byte chunk `ch` (0..15, or 0..7 for head_dim 64) of row r
// of a 128-row tile
__device__ __forceinline__ uint32_t sw_chunk(int r, int ch) {
    return (ch >> 3) * (128 * 128) + r * 128 + (((ch & 7) ^ (r & 7)) << 4);
}

__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((addr & 0x3FFFF) >> 4);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFF) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFF) << 32;
    d |= 1ull << 46;   // descriptor version
    d |= 2ull << 61;   // 128-byte swizzle
    return d;
}
// kind::f16 instruction descriptor: f32 accumulate, bf16 A and B
constexpr uint32_t idesc(int M, int N, int b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(b_mn_major) << 16) |
           (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void mma_f16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t id,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
        "l"(a), "l"(b), "r"(id), "r"(accumulate));
}
// descriptor from its halves (the low half holds the start address >> 4)
__device__ __forceinline__ uint64_t desc_at(uint32_t lo, uint32_t hi) {
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "r"(lo), "r"(hi));
    return d;
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(bar)
                 : "memory");
}
__device__ __forceinline__ bool bar_wait(uint32_t bar, uint32_t parity) {
    for (int i = 0; i < (1 << 20); ++i) {
        uint32_t ok;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
            " selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
        if (ok) return true;
    }
    return false;
}
// Packed fp32 pairs (two lanes of one 64-bit register; one instruction for
// both): the softmax issues one instruction where it issued two.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
    return d;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
// 2^x with the hardware approximation (flush-to-zero); 2^-inf = 0
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }

// 64 consecutive fp32 columns of this thread's TMEM lane; the wait is in the
// same asm block, so the values exist only once the load has completed
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&v)[64]) {
    uint32_t r[64];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];\n"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}
// 32 consecutive fp32 columns of this thread's TMEM lane (load and wait)
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
        "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
        "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
        "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
        "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
        "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31])));
}

// O (f32, TMEM) += A (bf16 pairs in TMEM, lane = row) x B (shared-memory descriptor)
__device__ __forceinline__ void mma_f16_ta(uint32_t tmem_d, uint32_t tmem_a, uint64_t b, uint32_t id,
                                           uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(tmem_d),
        "r"(tmem_a), "l"(b), "r"(id), "r"(accumulate));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count));
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void named_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(threads) : "memory");
}
__device__ __forceinline__ void tmem_st8u(uint32_t taddr, const uint32_t (&v)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};\n" ::"r"(taddr),
                 "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]));
}
// The order in which the prefill takes its entries, when the caller gives a
// workspace.  The hardware hands CTAs to SMs in launch order, and a CTA's
// work grows with its entry's kv_len (each of its query-tile pairs streams up
// to kv_len / 128 key tiles), so launching the entries by decreasing kv_len
// makes the list schedule longest first: the short entries fill the SMs at
// the end instead of a long one starting last.  One CTA: thread t checks
// entry t as the prefill kernel would (a failure is recorded here and the
// entry is ranked last, with no work), ranks it by (kv_len descending, entry
// ascending) against all entries, and writes its row of the table.  The
// prefill kernel is launched as this kernel's programmatic dependent and
// reads its row after griddepcontrol.wait.
constexpr int kPlanThreads = kPlanMaxBatch;

__global__ void __launch_bounds__(kPlanThreads) prefill_plan_kernel(const PrefillParams p) {
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    __shared__ int s_key[kPlanThreads];
    const int t = threadIdx.x;
    int r = 0, qo0 = 0, q_len = 0, kv_len = 0, key = -1;
    if (t < p.batch) {
        r = __ldg(p.req_pool_indices + t);
        qo0 = __ldg(p.qo_indptr + t);
        q_len = __ldg(p.qo_indptr + t + 1) - qo0;
        kv_len = __ldg(p.kv_indptr + t + 1) - __ldg(p.kv_indptr + t);
        const long long q_total = __ldg(p.qo_indptr + p.batch);
        const bool rows_ok = qo0 >= 0 && static_cast<long long>(qo0) + q_len <= q_total;
        if (static_cast<unsigned>(r) >= static_cast<unsigned>(p.num_reqs) || q_len < 0 || !rows_ok ||
            q_len > p.max_q_len || kv_len < q_len || kv_len > p.max_ctx_len || kv_len > p.max_kv_len)
            record_error(p.err, static_cast<unsigned>(r) >= static_cast<unsigned>(p.num_reqs) ? r
                                : (q_len >= 0 && !rows_ok) ? qo0 : kv_len);
        else
            key = kv_len;
    }
    s_key[t] = key;
    __syncthreads();
    if (t >= p.batch) return;
    int rank = 0;
    for (int e = 0; e < p.batch; ++e) {
        const int k = s_key[e];
        rank += k > key || (k == key && e < t);
    }
    int4 *row = reinterpret_cast<int4 *>(p.plan + 8 * rank);
    row[0] = make_int4(t, r, qo0, q_len);
    row[1] = make_int4(kv_len, key >= 0 ? 1 : 0, 0, 0);
}

// kGroup = false: the ragged prefill, one CTA per (query-tile pair, kv head,
// entry).  kGroup = true: the group role of a shared-prefix decode, one CTA
// per (chunk of the shared prefix, kv head, 256 query rows): the rows are the
// (entry b, head-in-group) pairs of the decode's q [batch, n_heads, D], the
// keys are the chunk's positions of the first entry's request row, nothing is
// masked, and the CTA ends with fp32 partials (o / l and (m, l)) that the
// decode's merge folds in.  Both share the pipeline below.
template <int G, bool kGroup, int D>
__global__ void __launch_bounds__(kNT, 1) prefill_tc_kernel(const PrefillParams p) {
    using bf16 = __nv_bfloat16;
    using L = TcLayout<D>;
    static_assert(!kGroup || D == 128, "the shared-prefix group role runs at head_dim 128");
    constexpr int kCR = L::kChunksRow, kChunks = L::kChunks, kTileBytes = L::kTileBytes;
    constexpr int kSmemQ = L::kSmemQ, kSmemK = L::kSmemK, kSmemV = L::kSmemV, kSmemBar = L::kSmemBar;
    constexpr int kSmemTmemAddr = L::kSmemTmemAddr, kSmemAbort = L::kSmemAbort, kSmemRed = L::kSmemRed;
    constexpr int kSmemSlots = L::kSmemSlots;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    const uint32_t s_base = smem_u32(sm);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + kSmemTmemAddr);
    volatile int *s_abort = reinterpret_cast<volatile int *>(sm + kSmemAbort);
    float *s_red = reinterpret_cast<float *>(sm + kSmemRed);
    auto bar = [&](int i) -> uint32_t { return s_base + kSmemBar + 8 * i; };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // The prefill launches the kv heads of one query-tile pair next to each
    // other (x), then the pairs (y, longest first), then the entries (z): the
    // CTAs running at once read the same token rows, each its head's part.
    const int g = kGroup ? static_cast<int>(blockIdx.y) : static_cast<int>(blockIdx.x);
    int qp, r, qo0, rows, kv_lo = 0, chunk = 0;
    int n_x[2], kv_end = 0;
    int lim_pos = 0;   // group: last key position of the chunk
    int P = 0;
    if constexpr (kGroup) {
        // the merge may launch now; it waits for this grid before reading
        asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
        chunk = blockIdx.x;
        qp = blockIdx.z;
        r = __ldg(p.req_pool_indices);   // the shared prefix is read from the first entry's row
        if (static_cast<unsigned>(r) >= static_cast<unsigned>(p.num_reqs)) {
            if (chunk == 0 && g == 0 && qp == 0 && tid == 0) record_error(p.err, r);
            r = 0;
        }
        qo0 = 0;
        rows = p.batch * G;
        kv_lo = chunk * p.chunk_len;
        kv_end = min(p.shared_len, kv_lo + p.chunk_len);
        lim_pos = kv_end - 1;
    } else {
        int q_len, kv_len;
        if (p.plan) {
            // the entry of rank blockIdx.z, longest first (checked by the plan kernel)
            asm volatile("griddepcontrol.wait;\n" ::: "memory");
            const int4 *row = reinterpret_cast<const int4 *>(p.plan) + 2 * blockIdx.z;
            const int4 e0 = __ldcg(row), e1 = __ldcg(row + 1);
            if (!e1.y) return;
            r = e0.y;
            qo0 = e0.z;
            q_len = e0.w;
            kv_len = e1.x;
        } else {
            const int b = blockIdx.z;
            r = __ldg(p.req_pool_indices + b);
            qo0 = __ldg(p.qo_indptr + b);
            q_len = __ldg(p.qo_indptr + b + 1) - qo0;
            kv_len = __ldg(p.kv_indptr + b + 1) - __ldg(p.kv_indptr + b);
            // q and o hold qo_indptr[batch] packed rows: this entry's rows must
            // lie inside them, or they are neither read nor written
            const long long q_total = __ldg(p.qo_indptr + p.batch);
            const bool rows_ok = qo0 >= 0 && static_cast<long long>(qo0) + q_len <= q_total;
            if (static_cast<unsigned>(r) >= static_cast<unsigned>(p.num_reqs) || q_len < 0 || !rows_ok ||
                q_len > p.max_q_len || kv_len < q_len || kv_len > p.max_ctx_len || kv_len > p.max_kv_len) {
                if (blockIdx.y == 0 && g == 0 && tid == 0)
                    record_error(p.err, static_cast<unsigned>(r) >= static_cast<unsigned>(p.num_reqs) ? r
                                        : (q_len >= 0 && !rows_ok) ? qo0 : kv_len);
                return;
            }
        }
        rows = q_len * G;
        P = kv_len - q_len;
        lim_pos = kv_len - 1;
        // the entry's pairs longest first, then the grid's spare pairs (no rows)
        qp = (rows + 2 * kRows - 1) / (2 * kRows) - 1 - static_cast<int>(blockIdx.y);
        if (qp < 0) return;
    }
    const int row0 = qp * 2 * kRows;
    if (row0 >= rows || kv_end - kv_lo < 0) return;
    // K/V tiles each query tile sees (0: the tile has no rows); B sees at least as many as A
#pragma unroll
    for (int X = 0; X < 2; ++X) {
        const int rx = row0 + X * kRows;
        n_x[X] = 0;
        if (rx < rows) {
            if constexpr (kGroup) {
                n_x[X] = (kv_end - kv_lo + kTok - 1) / kTok;
            } else {
                const int pos_last = (min(rx + kRows, rows) - 1) / G;
                const int e = p.causal ? min(lim_pos + 1, P + pos_last + 1) : lim_pos + 1;
                n_x[X] = (e + kTok - 1) / kTok;
                kv_end = max(kv_end, e);
            }
        }
    }
    const int n_tiles = max(n_x[0], n_x[1]);   // >= 1: kv_end > kv_lo when rows > 0
    if (n_tiles == 0) return;                  // an empty chunk (not launched by the host)

    const int64_t slot_stride = static_cast<int64_t>(p.n_kv_heads) * D;
    const bf16 *kbase = static_cast<const bf16 *>(p.k_buffer) + (p.layer_row0 * p.n_kv_heads + g) * D;
    const bf16 *vbase = static_cast<const bf16 *>(p.v_buffer) + (p.layer_row0 * p.n_kv_heads + g) * D;
    const int32_t *r2t = p.req_to_token + static_cast<int64_t>(r) * p.max_ctx_len;
    // slot of key position j (a page-table lookup in the group role when
    // page_size > 0); a slot or page outside the pool is recorded and read as 0
    auto slot_of = [&](int j) -> int {
        if (kGroup && p.page_size > 0) {
            const int pg = __ldg(p.req_to_page + static_cast<int64_t>(r) * p.max_pages + j / p.page_size);
            if (static_cast<unsigned long long>(static_cast<long long>(pg)) >=
                static_cast<unsigned long long>(p.n_pages)) {
                record_error(p.err, pg);
                return 0;
            }
            return pg * p.page_size + j % p.page_size;
        }
        int slot = __ldg(r2t + j);
        if (static_cast<unsigned long long>(static_cast<long long>(slot)) >=
            static_cast<unsigned long long>(p.size)) {
            record_error(p.err, slot);
            slot = 0;
        }
        return slot;
    };

    // ---- the prefill's producer (warps 8..14) gathers K/V tile t into ring
    // slot t % 2 through registers: the rows are mostly L2 hits here (each
    // request's K/V is read by all its query-tile pairs), where this measured
    // ~12% faster than the cp.async producer of the group role.  Tile t's
    // loads go out once tile t - 1 is stored, and tile 0's while the other
    // warps load the query tiles.
    const bool prefill_producer = !kGroup && warp >= kSoftmaxWarps && warp < kMmaWarp;
    const int pt = tid - kSoftmaxWarps * 32;
    int *s_slot = reinterpret_cast<int *>(sm + kSmemSlots);   // [2][kTok], by tile parity
    auto fetch = [&](int tile) -> int {   // slot of row pt of `tile`, -1 past the gathered range
        const int j = kv_lo + tile * kTok + pt;
        if (pt >= kTok || tile >= n_tiles || j >= kv_end) return -1;
        return slot_of(j);
    };
    uint4 kv[2][kChunks];   // the producer's tile in flight: K, V
    int slot_n = 0;         // the next tile's slot index (row pt), in flight
    auto stage_and_load = [&](int t) {
        int *slots = s_slot + (t & 1) * kTok;
        if (pt < kTok) slots[pt] = slot_n;
        slot_n = fetch(t + 1);
        named_sync(1, kPT);   // tile t's slots are staged
#pragma unroll
        for (int k = 0; k < kChunks; ++k) {
            const int i = pt + k * kPT;
            kv[0][k] = kv[1][k] = make_uint4(0u, 0u, 0u, 0u);
            if (i < kTok * kCR) {
                const int sl = slots[i / kCR];
                if (sl >= 0) {
                    const int64_t off = sl * slot_stride + (i % kCR) * 8;
                    kv[0][k] = __ldcg(reinterpret_cast<const uint4 *>(kbase + off));
                    kv[1][k] = __ldcg(reinterpret_cast<const uint4 *>(vbase + off));
                }
            }
        }
    };
    if (prefill_producer) {
        slot_n = fetch(0);
        stage_and_load(0);
    }

    // ---- setup: barriers, TMEM, the two query tiles
    if (tid == 0) {
        for (int i = 0; i < kNumBars; ++i) {
            uint32_t cnt = 1;
            if (i == kBarKFull || i == kBarKFull + 1 || i == kBarVFull || i == kBarVFull + 1) cnt = kPT;
            else if (i == kBarPFull || i == kBarPFull + 1) cnt = kSoftmaxWarps;
            mbar_init(bar(i), cnt);
        }
        *s_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
    }
    if (!prefill_producer) {
        // the softmax and MMA warps (all warps in the group role)
        const int qt = kGroup ? tid : (tid < kSoftmaxWarps * 32 ? tid : tid - kPT);
        const int qn = kGroup ? kNT : kNT - kPT;
        const bf16 *q = static_cast<const bf16 *>(p.q);
        for (int i = qt; i < 2 * kRows * kCR; i += qn) {
            const int X = i / (kRows * kCR), rr = (i / kCR) & (kRows - 1), ch = i % kCR;
            const int Rq = row0 + X * kRows + rr;
            void *dst = sm + kSmemQ + X * kTileBytes + sw_chunk(rr, ch);
            if (Rq < rows) {
                const int pos = Rq / G, hh = Rq - (Rq / G) * G;
                cp_async16(dst, q + ((static_cast<int64_t>(qo0) + pos) * p.n_heads + g * G + hh) * D + ch * 8);
            } else {
                cp_async16(dst, q, 0);
            }
        }
        cp_async_commit();
        cp_async_wait<0>();
    }
    fence_async_smem();
    fence_before();
    __syncthreads();   // barriers, the TMEM address and the query tiles are visible
    fence_after();
    const uint32_t tmem = *tmem_slot;

    if (prefill_producer) {
        // ================= producer (prefill): tile t is in registers (kv)
        // A wait that gives up sets the abort flag; after that nothing is
        // stored, but every producer barrier is still met.
        bool live = true;
        for (int t = 0; t < n_tiles; ++t) {
            live = live && *s_abort == 0 && bar_wait(bar(kBarKEmpty + (t & 1)), ((t >> 1) & 1) ^ 1);
#pragma unroll
            for (int X = 0; X < 2; ++X) {   // X = 0: K, 1: V
                if (X == 1) live = live && bar_wait(bar(kBarVEmpty + (t & 1)), ((t >> 1) & 1) ^ 1);
                if (!live) break;
                unsigned char *dst0 = sm + (X ? kSmemV : kSmemK) + (t & 1) * kTileBytes;
#pragma unroll
                for (int k = 0; k < kChunks; ++k) {
                    const int i = pt + k * kPT;
                    if (i < kTok * kCR) *reinterpret_cast<uint4 *>(dst0 + sw_chunk(i / kCR, i % kCR)) = kv[X][k];
                }
                fence_async_smem();   // these generic stores -> the tensor core's reads
                mbar_arrive(bar((X ? kBarVFull : kBarKFull) + (t & 1)));
            }
            if (!live && *s_abort == 0) {
                *s_abort = 1;
                record_error(p.err, -2001);
            }
            if (t + 1 < n_tiles) stage_and_load(t + 1);
        }
    } else if (warp >= kSoftmaxWarps && warp < kMmaWarp) {
        // ================= producer (group role): K and V tile t into ring slot t % 2.
        // The prefix rows come from DRAM while the private role streams at full
        // bandwidth, so load latency dominates: 16-byte cp.async copies straight into the swizzled ring (no
        // register round trip), so the copies of tile t are in flight while
        // those of tile t - 1 land.  Commit groups go K(0), V(0), K(1), V(1),
        // ...; once K(t) is committed, waiting until two groups remain means
        // K(t - 1) has landed (likewise V), and the thread then makes its
        // copies visible to the tensor core (proxy fence) and arrives on the
        // slot's full barrier.  K(t) waits for its slot to be released by
        // S(t - 2) and V(t) by P.V(t - 2), both of which the MMA thread can
        // issue without K(t - 1) or V(t - 1): no wait here depends on an
        // arrival that comes after it.
        auto issue = [&](int X, int t) {   // X = 0: K, 1: V; rows past the range are zero-filled
            const int *slots = s_slot + (t & 1) * kTok;
            unsigned char *dst0 = sm + (X ? kSmemV : kSmemK) + (t & 1) * kTileBytes;
            const bf16 *src0 = X ? vbase : kbase;
#pragma unroll
            for (int k = 0; k < kChunks; ++k) {
                const int i = pt + k * kPT;
                if (i < kTok * kCR) {
                    const int sl = slots[i / kCR];
                    void *dst = dst0 + sw_chunk(i / kCR, i % kCR);
                    if (sl >= 0) cp_async16(dst, src0 + sl * slot_stride + (i % kCR) * 8);
                    else cp_async16(dst, src0, 0);
                }
            }
            cp_async_commit();
        };
        auto publish = [&](int X, int t) {   // this thread's copies of tile t are complete
            fence_async_smem();
            mbar_arrive(bar((X ? kBarVFull : kBarKFull) + (t & 1)));
        };
        // A wait that gives up sets the abort flag; after that nothing is
        // issued or published, but every producer barrier is still met.
        slot_n = fetch(0);
        for (int t = 0; t < n_tiles; ++t) {
            int *slots = s_slot + (t & 1) * kTok;
            if (pt < kTok) slots[pt] = slot_n;
            slot_n = fetch(t + 1);   // the next tile's index is in flight meanwhile
            named_sync(1, kPT);      // this tile's slots are staged
            bool live = *s_abort == 0 && bar_wait(bar(kBarKEmpty + (t & 1)), ((t >> 1) & 1) ^ 1);
            if (live) issue(0, t);
            else cp_async_commit();
            cp_async_wait<2>();
            if (live && t > 0) publish(0, t - 1);
            live = live && bar_wait(bar(kBarVEmpty + (t & 1)), ((t >> 1) & 1) ^ 1);
            if (live) issue(1, t);
            else cp_async_commit();
            cp_async_wait<2>();
            if (live && t > 0) publish(1, t - 1);
            if (!live && *s_abort == 0) {
                *s_abort = 1;
                record_error(p.err, -2001);
            }
        }
        cp_async_wait<0>();
        if (*s_abort == 0) {
            publish(0, n_tiles - 1);
            publish(1, n_tiles - 1);
        }
    } else if (warp == kMmaWarp) {
        // ================= MMA issue
        if (lane == 0) {
            const uint32_t id_s = idesc(128, 128, 0), id_o = idesc(128, D, 1);
            // Descriptors are built once; a product's start address is a
            // 16-byte step added to the low half (every shared address is
            // below 2^18, so the 14-bit field cannot carry into the next).
            const uint64_t dq = sdesc(s_base + kSmemQ, 16, 1024), dk = sdesc(s_base + kSmemK, 16, 1024);
            const uint64_t dv = sdesc(s_base + kSmemV, 128 * 128, 1024);
            const uint32_t q_lo = static_cast<uint32_t>(dq), q_hi = static_cast<uint32_t>(dq >> 32);
            const uint32_t k_lo = static_cast<uint32_t>(dk), k_hi = static_cast<uint32_t>(dk >> 32);
            const uint32_t v_lo = static_cast<uint32_t>(dv), v_hi = static_cast<uint32_t>(dv >> 32);
            auto issue_s = [&](int X, int slot) {   // S_X = Q_X K^T
                const uint32_t qa = q_lo + X * (kTileBytes >> 4), ka = k_lo + slot * (kTileBytes >> 4);
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t off = ((ks >> 2) * (128 * 128) + (ks & 3) * 32) >> 4;
                    mma_f16(tmem + X * 256, desc_at(qa + off, q_hi), desc_at(ka + off, k_hi), id_s, ks > 0);
                }
                mma_commit(bar(kBarSFull + X));
            };
            auto issue_pv = [&](int X, int slot, bool acc) {   // O_X += P_X V; P over S_X's columns
                const uint32_t va = v_lo + slot * (kTileBytes >> 4);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    // tokens [16 ks, 16 ks + 16): half ks / 4 of the row, packed at its first 32 columns
                    const uint32_t pcol = (ks >> 2) * 64 + (ks & 3) * 8;
                    mma_f16_ta(tmem + X * 256 + 128, tmem + X * 256 + pcol, desc_at(va + ks * (16 * 128 >> 4), v_hi),
                               id_o, (acc || ks > 0) ? 1u : 0u);
                }
            };
            auto give_up = [&](int code) {
                *s_abort = 1;
                record_error(p.err, code);
            };
            // Waits for the K/V ring.  The prefill's producer stores tile t
            // once P.V_B(t - 2) has released its V slot, and each of its
            // threads arrives on K(t) full before V(t) full, so a complete
            // V(t) barrier means K(t) has landed too: one wait per tile,
            // made before S(t).  The group role's producer publishes V(t)
            // only after P.V_B(t - 1), which is issued after S(t): there S(t)
            // waits for K(t) and P.V(t) for V(t).
            auto wait_kv = [&](int t) -> bool {
                const uint32_t par = (t >> 1) & 1;
                return bar_wait(bar((kGroup ? kBarKFull : kBarVFull) + (t & 1)), par);
            };
            bool ok = wait_kv(0);
            if (!ok) give_up(-3002);
            if (ok) {
                fence_after();
                issue_s(0, 0);
                if (n_x[1] > 0) issue_s(1, 0);
                mma_commit(bar(kBarKEmpty));
            }
            for (int j = 0; ok && j < n_tiles; ++j) {
                if (*s_abort) break;
                const bool more = j + 1 < n_tiles;
                if (kGroup && !bar_wait(bar(kBarVFull + (j & 1)), (j >> 1) & 1)) { give_up(-3003); break; }
                if (j < n_x[0]) {
                    if (!bar_wait(bar(kBarPFull), j & 1)) { give_up(-3004); break; }
                    fence_after();
                    issue_pv(0, j & 1, j > 0);
                    if (j == n_x[0] - 1) mma_commit(bar(kBarODone));
                }
                if (more) {
                    if (!wait_kv(j + 1)) { give_up(-3005); break; }
                    fence_after();
                    if (j + 1 < n_x[0]) issue_s(0, (j + 1) & 1);
                }
                if (j < n_x[1]) {
                    if (!bar_wait(bar(kBarPFull + 1), j & 1)) { give_up(-3006); break; }
                    fence_after();
                    issue_pv(1, j & 1, j > 0);
                    if (j == n_x[1] - 1) mma_commit(bar(kBarODone + 1));
                }
                mma_commit(bar(kBarVEmpty + (j & 1)));
                if (more) {
                    if (j + 1 < n_x[1]) issue_s(1, (j + 1) & 1);
                    mma_commit(bar(kBarKEmpty + ((j + 1) & 1)));
                }
            }
        }
        __syncwarp();
    } else {
        // ================= softmax: row `row`, columns [64 hc, 64 hc + 64) of each tile
        if constexpr (kGroup) {
            // The statement that the prefix is shared: every other entry of
            // this CTA's rows must hold the first entry's table entries over
            // the chunk (its page ids, or its slots through req_to_token).  The
            // units to compare are split over the kv-head CTAs of the chunk; a
            // mismatch is recorded as -100000 - b.  These warps would
            // otherwise wait for the first scores.
            const int HK = p.n_kv_heads;
            const int b_lo = max(1, row0 / G), b_hi = min(p.batch, (row0 + 2 * kRows) / G);
            const int ps = p.page_size;
            const int u_lo = ps > 0 ? kv_lo / ps : kv_lo;
            const int u_hi = ps > 0 ? (kv_end - 1) / ps + 1 : kv_end;
            const int n_u = u_hi - u_lo > g ? (u_hi - u_lo - g + HK - 1) / HK : 0;
            const int n_b = max(0, b_hi - b_lo);
            const int32_t *tab = ps > 0 ? p.req_to_page : p.req_to_token;
            const int64_t pitch = ps > 0 ? p.max_pages : p.max_ctx_len;
            for (int i = tid; i < n_b * n_u; i += kSoftmaxWarps * 32) {
                const int b = b_lo + i / n_u, u = u_lo + g + HK * (i % n_u);
                const int rb = __ldg(p.req_pool_indices + b);
                if (static_cast<unsigned>(rb) >= static_cast<unsigned>(p.num_reqs)) {
                    record_error(p.err, rb);
                    continue;
                }
                if (__ldg(tab + rb * pitch + u) != __ldg(tab + r * pitch + u)) record_error(p.err, -100000 - b);
            }
        }
        const int row = (warp & 3) * 32 + lane;   // TMEM lane = query row of this thread
        const int hc = warp >> 2;                  // column half
        const int pair_bar = 2 + (warp & 3);       // named barrier of warps w and w + 4
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const float sc = p.scale_log2;
        float m_run[2] = {-INFINITY, -INFINITY}, l_part[2] = {0.f, 0.f};   // l: this half's columns
        int lim[2];
#pragma unroll
        for (int X = 0; X < 2; ++X) {
            const int R = row0 + X * kRows + row;
            lim[X] = R < rows ? ((!kGroup && p.causal) ? P + R / G : lim_pos) : -1;   // last visible position
        }
        // A wait that gives up sets the abort flag; after that no wait is made,
        // but every named barrier is still met so the pair stays in step.
        auto wait_ok = [&](uint32_t br, uint32_t par) -> bool {
            bool ok = *s_abort == 0 && bar_wait(br, par);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok && lane == 0 && *s_abort == 0) {
                *s_abort = 1;
                record_error(p.err, -2007);
            }
            return ok;
        };
        for (int j = 0; j < n_tiles; ++j) {
#pragma unroll
            for (int X = 0; X < 2; ++X) {
                if (j >= n_x[X]) continue;   // CTA-uniform
                wait_ok(bar(kBarSFull + X), j & 1);
                fence_after();
                const uint32_t tS = tmem + X * 256 + lane_off + hc * 64;
                const int jt = kv_lo + j * kTok + hc * 64;
                // this half's 64 scores, read once; masked only near the diagonal
                float sv[64];
                tmem_ld64(tS, sv);
                if (jt + 63 > lim[X]) {
#pragma unroll
                    for (int i = 0; i < 64; ++i)
                        if (jt + i > lim[X]) sv[i] = -INFINITY;
                }
                float mx[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) mx[u] = -INFINITY;
#pragma unroll
                for (int i = 0; i < 64; i += 2) mx[(i >> 1) & 7] = max3(mx[(i >> 1) & 7], sv[i], sv[i + 1]);
                float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                 fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) * sc;   // -inf stays -inf
                float *red = s_red + (X * 2 + (j & 1)) * 2 * kRows;
                red[hc * kRows + row] = mt;
                named_sync(pair_bar, 64);
                mt = fmaxf(mt, red[(hc ^ 1) * kRows + row]);
                // Raise the reference only when the tile maximum exceeds it by
                // more than 2^8, so P stays <= 2^8 and O is rescaled rarely.  TMEM
                // access is warp-collective: a warp rescales if any row must.
                const bool raise = mt > m_run[X] + kRescale || (m_run[X] == -INFINITY && mt != -INFINITY);
                const float alpha = raise ? exp2f(m_run[X] - mt) : 1.f;   // 0 on the first visible tile
                const bool touch_o = raise && j > 0 && m_run[X] != -INFINITY;
                if (__any_sync(0xffffffffu, touch_o)) {
                    const float f = touch_o ? alpha : 1.f;
                    const uint32_t tO = tmem + X * 256 + 128 + lane_off + hc * (D / 2);
#pragma unroll 1
                    for (int h2 = 0; h2 < D / 64; ++h2) {   // one 32-column piece at a time: sv stays live
                        float v[32];
                        tmem_ld32(tO + h2 * 32, v);
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] *= f;
                        tmem_st32(tO + h2 * 32, v);
                    }
                }
                if (raise) {
                    l_part[X] *= alpha;
                    m_run[X] = mt;
                }
                // P = 2^(s - m) as bf16 pairs over the first 32 of this half's S
                // columns (already read); a row with nothing visible yet keeps
                // P = 0 (reference -inf, fma(v, scale, -inf) = -inf for finite
                // or -inf v)
                const float neg_m = m_run[X] == -INFINITY ? -INFINITY : -m_run[X];
                // the exponents and the row sum two lanes at a time (packed fp32)
                const uint64_t sc2 = f2_pack(sc, sc), nm2 = f2_pack(neg_m, neg_m);
                uint64_t ls2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t pk[8];
#pragma unroll
                    for (int i = 0; i < 16; i += 2) {
                        float x0, x1;
                        f2_unpack(f2_fma(f2_pack(sv[c * 16 + i], sv[c * 16 + i + 1]), sc2, nm2), x0, x1);
                        const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                        ls2[(i >> 1) & 3] = f2_add(ls2[(i >> 1) & 3], f2_pack(p0, p1));
                        __nv_bfloat162 h = __floats2bfloat162_rn(p0, p1);
                        pk[i >> 1] = *reinterpret_cast<uint32_t *>(&h);
                    }
                    tmem_st8u(tS + c * 8, pk);
                }
                float l0, l1, l2, l3, l4, l5, l6, l7;
                f2_unpack(ls2[0], l0, l1);
                f2_unpack(ls2[1], l2, l3);
                f2_unpack(ls2[2], l4, l5);
                f2_unpack(ls2[3], l6, l7);
                l_part[X] += ((l0 + l1) + (l2 + l3)) + ((l4 + l5) + (l6 + l7));
                asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
                fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(kBarPFull + X));   // P_X(j) and the rescaled O_X ready
            }
        }
        // ---- epilogue: O_X is final once its last P.V is done
#pragma unroll
        for (int X = 0; X < 2; ++X) {
            if (n_x[X] == 0) continue;
            const bool done = wait_ok(bar(kBarODone + X), 0);
            fence_after();
            float *red = s_red + (X * 2 + (n_x[X] & 1)) * 2 * kRows;   // the buffer the last tile did not use
            red[hc * kRows + row] = l_part[X];
            named_sync(pair_bar, 64);
            const float l_row = l_part[X] + red[(hc ^ 1) * kRows + row];
            const float inv = l_row > 0.f ? 1.f / l_row : 0.f;
            const int R = row0 + X * kRows + row;
            const int pos = R / G, hh = R - (R / G) * G;
            const bool store = done && *s_abort == 0 && R < rows;
            if constexpr (kGroup) {
                // fp32 partial of entry pos, head g G + hh: o / l, then (m, l).
                // The warp's 32 rows x 64 columns go through shared memory (the
                // query and K tiles, whose last reader -- the final S product
                // -- completed before this tile's O) so that global stores
                // write whole 256-byte row pieces instead of one row per lane.
                const uint64_t pol = l2_keep_policy();
                float *stg = reinterpret_cast<float *>(sm + kSmemQ) + warp * 32 * kStgPitch;
#pragma unroll
                for (int c0 = 0; c0 < 64; c0 += 32) {
                    float ov[32];
                    tmem_ld32(tmem + X * 256 + 128 + lane_off + hc * 64 + c0, ov);
#pragma unroll
                    for (int q4 = 0; q4 < 8; ++q4)
                        *reinterpret_cast<float4 *>(stg + lane * kStgPitch + c0 + 4 * q4) =
                            make_float4(ov[4 * q4] * inv, ov[4 * q4 + 1] * inv, ov[4 * q4 + 2] * inv,
                                        ov[4 * q4 + 3] * inv);
                }
                __syncwarp();
                if (done && *s_abort == 0) {
                    // two rows per instruction, 16 lanes x 16 bytes each
#pragma unroll 4
                    for (int i = 0; i < 16; ++i) {
                        const int rr = 2 * i + (lane >> 4), ch = lane & 15;
                        const int Rr = row0 + X * kRows + (warp & 3) * 32 + rr;
                        if (Rr < rows) {
                            const int64_t unit_r = p.unit0 +
                                (static_cast<int64_t>(chunk) * p.batch + Rr / G) * p.n_heads + g * G + Rr % G;
                            const float4 v = *reinterpret_cast<const float4 *>(stg + rr * kStgPitch + ch * 4);
                            st_keep4(p.o_part + unit_r * D + hc * 64 + ch * 4, v.x, v.y, v.z, v.w, pol);
                        }
                    }
                }
                __syncwarp();   // the staging rows are rewritten for the next tile
                if (store && hc == 0) {
                    const int64_t unit =
                        p.unit0 + (static_cast<int64_t>(chunk) * p.batch + pos) * p.n_heads + g * G + hh;
                    st_keep(p.ml_part + unit * 2, m_run[X], pol);
                    st_keep(p.ml_part + unit * 2 + 1, l_row, pol);
                }
            } else {
                // The warp's 32 rows x D/2 columns go through shared memory so
                // that global stores write whole row halves (8, or 4 at head_dim
                // 64, lanes per row) instead of one row per lane.  The staging
                // is the first query tile's area: its last S product completed
                // before O_A, tile B's epilogue comes after tile A's, and 16-byte
                // chunk c of row r sits at chunk c ^ (r % kCH) (no bank conflicts).
                constexpr int kCH = D / 16;              // 16-byte chunks per row half
                constexpr int kRowB = D;                 // bytes per staged row half
                unsigned char *stg = sm + kSmemQ + warp * 32 * kRowB;
#pragma unroll
                for (int c0 = 0; c0 < D / 2; c0 += 32) {
                    float ov[32];
                    tmem_ld32(tmem + X * 256 + 128 + lane_off + hc * (D / 2) + c0, ov);
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 32; i += 2) {
                        __nv_bfloat162 h = __floats2bfloat162_rn(ov[i] * inv, ov[i + 1] * inv);
                        pk[i >> 1] = *reinterpret_cast<uint32_t *>(&h);
                    }
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        const int c = c0 / 8 + q4;
                        *reinterpret_cast<uint4 *>(stg + lane * kRowB + ((c ^ (lane % kCH)) << 4)) =
                            make_uint4(pk[4 * q4], pk[4 * q4 + 1], pk[4 * q4 + 2], pk[4 * q4 + 3]);
                    }
                }
                __syncwarp();
                if (done && *s_abort == 0) {
                    // rows past the request are not stored
#pragma unroll
                    for (int i = 0; i < kCH; ++i) {
                        const int rr = i * (32 / kCH) + lane / kCH, c = lane % kCH;
                        const int Rr = row0 + X * kRows + (warp & 3) * 32 + rr;
                        if (Rr < rows) {
                            const int pr = Rr / G, hr = Rr - (Rr / G) * G;
                            bf16 *dst = static_cast<bf16 *>(p.o) +
                                        ((static_cast<int64_t>(qo0) + pr) * p.n_heads + g * G + hr) * D + hc * (D / 2) +
                                        c * 8;
                            *reinterpret_cast<uint4 *>(dst) =
                                *reinterpret_cast<const uint4 *>(stg + rr * kRowB + ((c ^ (rr % kCH)) << 4));
                        }
                    }
                }
                __syncwarp();   // the staging rows are rewritten for the next tile
            }
        }
    }
    fence_before();
    __syncthreads();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(kTmemCols));
    if constexpr (kGroup) {
        // This grid was launched as a programmatic dependent of the decode's
        // split kernel (the private role): it completes only after that one,
        // so the merge, which waits for this grid, sees both roles' partials.
        asm volatile("griddepcontrol.wait;\n" ::: "memory");
    }
}

template <int G, bool kGroup, int D>
cudaError_t set_smem_once() {
    static std::atomic<uint64_t> attr_done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(attr_done.load() & bit)) {
        e = cudaFuncSetAttribute(prefill_tc_kernel<G, kGroup, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 TcLayout<D>::kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_done.fetch_or(bit);
    }
    return cudaSuccess;
}

template <int G, int D>
cudaError_t run(const PrefillParams &p, cudaStream_t s) {
    cudaError_t e = set_smem_once<G, false, D>();
    if (e != cudaSuccess) return e;
    const int qtiles = (p.max_q_len * G + kRows - 1) / kRows;
    const dim3 grid(p.n_kv_heads, (qtiles + 1) / 2, p.batch);   // two query tiles per CTA, heads fastest
    if (!p.plan) {
        prefill_tc_kernel<G, false, D><<<grid, kNT, TcLayout<D>::kSmemBytes, s>>>(p);
        return cudaGetLastError();
    }
    // the entry order first; the prefill as its programmatic dependent
    prefill_plan_kernel<<<1, kPlanThreads, 0, s>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kNT);
    cfg.dynamicSmemBytes = TcLayout<D>::kSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, prefill_tc_kernel<G, false, D>, p);
}

template <int D>
cudaError_t run_d(const PrefillParams &p, int group, cudaStream_t s) {
    switch (group) {
        case 1: return run<1, D>(p, s);
        case 2: return run<2, D>(p, s);
        case 4: return run<4, D>(p, s);
        case 8: return run<8, D>(p, s);
        default: return cudaErrorNotSupported;
    }
}

template <int G>
cudaError_t run_group(const DecodeParams &d, cudaStream_t s) {
    cudaError_t e = set_smem_once<G, true, 128>();
    if (e != cudaSuccess) return e;
    PrefillParams p{};
    p.q = d.q;
    p.k_buffer = d.k_buffer;
    p.v_buffer = d.v_buffer;
    p.req_to_token = d.req_to_token;
    p.req_pool_indices = d.req_pool_indices;
    p.size = d.size;
    p.layer_row0 = d.layer_row0;
    p.n_kv_heads = d.n_kv_heads;
    p.n_heads = d.n_heads;
    p.num_reqs = d.num_reqs;
    p.max_ctx_len = d.max_ctx_len;
    p.batch = d.batch;
    p.scale_log2 = d.scale_log2;
    p.err = d.err;
    p.req_to_page = d.req_to_page;
    p.max_pages = d.max_pages;
    p.page_size = d.page_size;
    p.n_pages = d.n_pages;
    p.shared_len = d.shared_len;
    p.chunk_len = d.group_chunk_len;
    p.o_part = d.o_part;
    p.ml_part = d.ml_part;
    p.unit0 = d.group_unit0;
    const int row_blocks = (d.batch * G + kGroupRows - 1) / kGroupRows;
    // a programmatic dependent of the split kernel: its CTAs start on the SMs
    // the split kernel leaves free, without waiting for it to finish
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(d.group_chunks, d.n_kv_heads, row_blocks);
    cfg.blockDim = dim3(kNT);
    cfg.dynamicSmemBytes = TcLayout<128>::kSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, prefill_tc_kernel<G, true, 128>, p);
}

}  // namespace

bool prefill_supported(int dtype, int head_dim, int group) {
    return dtype == PKV_BF16 && (head_dim == 64 || head_dim == 128) &&
           (group == 1 || group == 2 || group == 4 || group == 8);
}

cudaError_t launch_prefill(const PrefillParams &p, int dtype, int head_dim, int group, cudaStream_t s) {
    if (!prefill_supported(dtype, head_dim, group)) return cudaErrorNotSupported;
    if (p.batch == 0 || p.max_q_len == 0) return cudaSuccess;
    PrefillParams q = p;
    if (q.batch < 2 || q.batch > kPlanMaxBatch) q.plan = nullptr;
    return head_dim == 128 ? run_d<128>(q, group, s) : run_d<64>(q, group, s);
}

cudaError_t launch_shared_group_tc(const DecodeParams &p, int group, cudaStream_t s) {
    switch (group) {
        case 1: return run_group<1>(p, s);
        case 2: return run_group<2>(p, s);
        case 4: return run_group<4>(p, s);
        case 8: return run_group<8>(p, s);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace pkv
