// pkv_prefill_tc.cu -- ragged paged prefill on the 5th-generation tensor cores
// (tcgen05, accumulators in tensor memory), bf16, head_dim 128.
//
// Operation: as in pkv_prefill.cu (AstrAI docs/guides/inference.md,
// "Attention Backend" prefill path; causal alignment from
// astrai/model/transformer.py process_attention_mask): packed query row
// qo_indptr[b] + i, head h attends to slots req_to_token[req_pool_indices[b], j]
// for j <= P + i (P = kv_len - q_len) or j < kv_len when not causal.
//
// One CTA of 8 warps per (query tile, kv head, entry).  A query tile is 128
// rows of (position, head-in-group) pairs, so the G query heads of a kv head
// share every gathered K/V tile; warps w and w+4 share TMEM lanes 32(w%4)..
// and split each row's columns in halves.  TMEM holds two S buffers and O, so
// the tensor core computes S_{j+1} (and then P.V_j) while the threads run the
// softmax of tile j.  Per 128-token K/V tile j:
//   1. wait S_j (tcgen05.commit -> mbarrier), issue S_{j+1} = Q K_{j+1}^T
//      (8 tcgen05.mma, M=128, N=128, K=16) into the other S buffer, and start
//      gathering K_{j+2} (cp.async, slot indices staged in shared memory from
//      a register prefetched ahead) into the K slot S_j just released;
//   2. softmax: thread r reads its row of S_j with tcgen05.ld, keeps a running
//      maximum that is only raised when the tile maximum exceeds it by more
//      than 2^8 (then O and l are rescaled in TMEM, after P.V_{j-1} is done),
//      and writes P = 2^(s - m) as bf16 into a 128-byte-swizzled K-major tile;
//      V_{j+1} is gathered into the V slot P.V_{j-1} released;
//   3. O += P V_j: 8 tcgen05.mma (V read MN-major) into TMEM.
// Operand tiles use the 128-byte swizzle: a [rows x 128] bf16 tile is two
// 64-column halves of rows x 128 B, 16-byte chunk c of row r stored at chunk
// c ^ (r % 8), atoms 1024-byte aligned.  Every mbarrier wait is bounded.
#include <atomic>

#include "pkv_common.cuh"
#include "pkv_launch.h"

namespace pkv {
namespace {

constexpr int kRows = 128;       // query rows per CTA (TMEM lanes)
constexpr int kTok = 128;        // kv tokens per tile
constexpr int kD = 128;
constexpr int kNT = 256;         // 8 warps: two threads per row, 64 columns each
constexpr int kTileBytes = 128 * 128 * 2;                 // 32 KB: any [128 x 128] bf16 tile
constexpr int kSmemQ = 0;
constexpr int kSmemK = kTileBytes;                        // [2 slots] K tiles
constexpr int kSmemV = kSmemK + 2 * kTileBytes;           // [2 slots] V tiles
constexpr int kSmemP = kSmemV + 2 * kTileBytes;
constexpr int kSmemBar = kSmemP + kTileBytes;             // mbarriers + tmem address
constexpr int kSmemSlots = kSmemBar + 64;                 // [4][kTok] int slots of tiles
constexpr int kSmemRed = kSmemSlots + 4 * 128 * 4;        // [2][kRows] float
constexpr int kSmemBytes = kSmemRed + 2 * 128 * 4 + 1024; // + alignment slack
constexpr uint32_t kTmemCols = 512;                       // S0: 0..127, S1: 128..255, O: 256..383
constexpr float kRescale = 8.f;                           // lazy rescale threshold (log2 units)

// byte offset of 16-byte chunk `ch` (0..15) of row r
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

template <int G>
__global__ void __launch_bounds__(kNT, 1) prefill_tc_kernel(const PrefillParams p) {
    using bf16 = __nv_bfloat16;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    const uint32_t s_base = smem_u32(sm);
    // bars[0], bars[1]: S buffer 0 / 1 complete; bars[2]: O (P.V) complete
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + kSmemBar);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + kSmemBar + 32);
    int *s_slot = reinterpret_cast<int *>(sm + kSmemSlots);          // [4][kTok]: tile t at t % 4
    float *s_red = reinterpret_cast<float *>(sm + kSmemRed);         // [2 halves][kRows]

    const int b = blockIdx.z, g = blockIdx.y;
    const int qt = gridDim.x - 1 - blockIdx.x;   // longest causal work first
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int row = (warp & 3) * 32 + lane;     // TMEM lane = query row of this thread
    const int hc = warp >> 2;                    // column half this thread handles

    int r = __ldg(p.req_pool_indices + b);
    const int qo0 = __ldg(p.qo_indptr + b);
    const int q_len = __ldg(p.qo_indptr + b + 1) - qo0;
    const int kv_len = __ldg(p.kv_indptr + b + 1) - __ldg(p.kv_indptr + b);
    if (static_cast<unsigned>(r) >= static_cast<unsigned>(p.num_reqs) || q_len < 0 ||
        q_len > p.max_q_len || kv_len < q_len || kv_len > p.max_ctx_len || kv_len > p.max_kv_len) {
        if (qt == 0 && g == 0 && tid == 0)
            record_error(p.err, static_cast<unsigned>(r) >= static_cast<unsigned>(p.num_reqs) ? r : kv_len);
        return;
    }
    const int rows = q_len * G;
    const int row0 = qt * kRows;
    if (row0 >= rows) return;
    const int P = kv_len - q_len;
    const int pos_last = (min(row0 + kRows, rows) - 1) / G;
    const int kv_end = p.causal ? min(kv_len, P + pos_last + 1) : kv_len;
    const int n_tiles = (kv_end + kTok - 1) / kTok;

    const int64_t slot_stride = static_cast<int64_t>(p.n_kv_heads) * kD;
    const bf16 *kbase = static_cast<const bf16 *>(p.k_buffer) + (p.layer_row0 * p.n_kv_heads + g) * kD;
    const bf16 *vbase = static_cast<const bf16 *>(p.v_buffer) + (p.layer_row0 * p.n_kv_heads + g) * kD;
    const int32_t *r2t = p.req_to_token + static_cast<int64_t>(r) * p.max_ctx_len;

    // slot of token tid of tile `tile` (threads 0..kTok-1), 0 past the visible range
    auto fetch_slot = [&](int tile) -> int {
        const int j = tile * kTok + tid;
        if (tid >= kTok || tile >= n_tiles || j >= kv_end) return 0;
        int slot = __ldg(r2t + j);
        if (static_cast<unsigned long long>(static_cast<long long>(slot)) >=
            static_cast<unsigned long long>(p.size)) {
            record_error(p.err, slot);
            slot = 0;
        }
        return slot;
    };
    // gather K (is_v = 0) or V rows of tile `tile` into ring slot tile % 2
    auto load_tile = [&](int tile, int is_v) {
        const int j0 = tile * kTok;
        const int *slots = s_slot + (tile & 3) * kTok;
        unsigned char *dst0 = sm + (is_v ? kSmemV : kSmemK) + (tile & 1) * kTileBytes;
        const bf16 *base = is_v ? vbase : kbase;
#pragma unroll 8
        for (int i = tid; i < kTok * 16; i += kNT) {
            const int t = i >> 4, ch = i & 15;
            void *dst = dst0 + sw_chunk(t, ch);
            if (j0 + t < kv_end)
                cp_async16(dst, base + slots[t] * slot_stride + ch * 8);
            else
                cp_async16(dst, kbase, 0);
        }
    };
    auto issue_s = [&](int tile) {   // thread 0: S[tile % 2] = Q K_tile^T
        fence_after();
        const uint32_t kaddr = s_base + kSmemK + (tile & 1) * kTileBytes;
        const uint32_t id_s = idesc(128, 128, 0);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            const uint32_t off = (ks >> 2) * (128 * 128) + (ks & 3) * 32;
            mma_f16(*tmem_slot + (tile & 1) * 128, sdesc(s_base + kSmemQ + off, 16, 1024),
                    sdesc(kaddr + off, 16, 1024), id_s, ks > 0);
        }
        mma_commit(smem_u32(bars + (tile & 1)));
    };

    // ---- prologue: slots of tiles 0..2, Q + K0, K1, V0
    if (tid < kTok) {
        s_slot[tid] = fetch_slot(0);
        s_slot[kTok + tid] = fetch_slot(1);
        s_slot[2 * kTok + tid] = fetch_slot(2);
    }
    int slot_next = fetch_slot(3);
    if (tid == 0) {
        for (int i = 0; i < 3; ++i)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(smem_u32(bars + i)));
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
    }
    {
        const bf16 *q = static_cast<const bf16 *>(p.q);
        for (int i = tid; i < kRows * 16; i += kNT) {
            const int rr = i >> 4, ch = i & 15;
            const int Rq = row0 + rr;
            void *dst = sm + kSmemQ + sw_chunk(rr, ch);
            if (Rq < rows) {
                const int pos = Rq / G, hh = Rq - (Rq / G) * G;
                cp_async16(dst, q + ((static_cast<int64_t>(qo0) + pos) * p.n_heads + g * G + hh) * kD + ch * 8);
            } else {
                cp_async16(dst, q, 0);
            }
        }
    }
    fence_before();
    __syncthreads();   // slots of tiles 0..2 and the TMEM address are visible
    fence_after();
    load_tile(0, 0);
    cp_async_commit();            // group: Q + K0
    if (n_tiles > 1) load_tile(1, 0);
    cp_async_commit();            // group: K1
    load_tile(0, 1);
    cp_async_commit();            // group: V0
    cp_async_wait<0>();
    fence_async_smem();
    __syncthreads();
    if (tid == 0) issue_s(0);

    const uint32_t tmem = *tmem_slot;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;   // this warp's TMEM lanes
    const uint32_t tO = tmem + 256 + lane_off + hc * 64;
    const int R = row0 + row;
    const int lim = R < rows ? (p.causal ? P + R / G : kv_len - 1) : -1;   // last visible position
    float m_run = -INFINITY, l_part = 0.f;   // l_part: this thread's 64 columns only
    bool ok = true;
    const uint32_t id_o = idesc(128, 128, 1);

    // Iteration j: S_j is in flight (or done); the tensor core queue is
    // [.. S_j, P.V_{j-1}]; we add S_{j+1} before the softmax of tile j.
    for (int j = 0; j < n_tiles && ok; ++j) {
        const uint32_t tS = tmem + (j & 1) * 128 + lane_off + hc * 64;
        // K_{j+1} (group issued one iteration ago) must have landed for S_{j+1}
        if (j >= 1) cp_async_wait<1>();
        fence_async_smem();
        // S_j complete: the threads may read it; its K slot is free.
        ok = __syncthreads_and(bar_wait(smem_u32(bars + (j & 1)), (j >> 1) & 1)) != 0;
        fence_after();
        if (!ok) break;
        if (tid == 0 && j + 1 < n_tiles) issue_s(j + 1);
        // next tiles' slots and the K_{j+2} gather (into the slot S_j just freed)
        if (tid < kTok) s_slot[((j + 3) & 3) * kTok + tid] = slot_next;
        slot_next = fetch_slot(j + 4);
        if (j + 2 < n_tiles) load_tile(j + 2, 0);
        cp_async_commit();        // group A_j: K_{j+2}

        // ---- softmax: this thread's row, columns [64 hc, 64 hc + 64)
        const int jt = j * kTok + hc * 64;
        const bool need_mask = jt + 63 > lim;
        float sv[64];   // this thread's 64 scores, read once
        tmem_ld64(tS, sv);
        if (need_mask) {
#pragma unroll
            for (int i = 0; i < 64; ++i)
                if (jt + i > lim) sv[i] = -INFINITY;
        }
        float mx[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) mx[u] = -INFINITY;
#pragma unroll
        for (int i = 0; i < 64; ++i) mx[i & 7] = fmaxf(mx[i & 7], sv[i]);
        const float mraw = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                 fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
        float mt = mraw * p.scale_log2;   // -inf stays -inf
        s_red[hc * kRows + row] = mt;
        // P.V_{j-1} must be complete before O is rescaled and P is rewritten;
        // then its V slot takes V_{j+1}.
        const bool o_ok = j == 0 || bar_wait(smem_u32(bars + 2), (j - 1) & 1);
        ok = __syncthreads_and(o_ok) != 0;
        fence_after();
        if (!ok) break;
        if (j + 1 < n_tiles) load_tile(j + 1, 1);
        cp_async_commit();        // group B_j: V_{j+1}
        mt = fmaxf(mt, s_red[(hc ^ 1) * kRows + row]);
        // Raise the reference only when the tile maximum exceeds it by more than
        // 2^8, so that P stays <= 2^8 and O is rescaled rarely.  TMEM accesses
        // are warp-collective: a warp rescales if any of its rows must.
        const bool raise = mt > m_run + kRescale || (m_run == -INFINITY && mt != -INFINITY);
        const float alpha = raise ? exp2f(m_run - mt) : 1.f;   // 0 on the first visible tile
        const bool touch_o = raise && j > 0 && m_run != -INFINITY;
        if (__any_sync(0xffffffffu, touch_o)) {
            const float f = touch_o ? alpha : 1.f;
            float ov[64];
            tmem_ld64(tO, ov);
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                float v[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = ov[h2 * 32 + i] * f;
                tmem_st32(tO + h2 * 32, v);
            }
            asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
        }
        if (raise) {
            l_part *= alpha;
            m_run = mt;
        }
        float ls[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        // a row with nothing visible yet keeps P = 0: its reference is -inf and
        // fma(v, scale, -inf) = -inf for finite or -inf v
        const float neg_m = m_run == -INFINITY ? -INFINITY : -m_run;
        const float sc = p.scale_log2;
#pragma unroll
        for (int c0 = 0; c0 < 64; c0 += 32) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
                const float p0 = ex2_approx(fmaf(sv[c0 + i], sc, neg_m));
                const float p1 = ex2_approx(fmaf(sv[c0 + i + 1], sc, neg_m));
                ls[(i >> 1) & 7] += p0 + p1;
                __nv_bfloat162 h = __floats2bfloat162_rn(p0, p1);
                pk[i >> 1] = *reinterpret_cast<uint32_t *>(&h);
            }
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
                *reinterpret_cast<uint4 *>(sm + kSmemP + sw_chunk(row, hc * 8 + (c0 >> 3) + q4)) =
                    make_uint4(pk[4 * q4], pk[4 * q4 + 1], pk[4 * q4 + 2], pk[4 * q4 + 3]);
        }
        l_part += ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
        // V_j (group B_{j-1}) must have landed: newer groups are A_j and B_j
        cp_async_wait<2>();
        fence_async_smem();   // P and V_j (generic writes) -> visible to the tensor core
        fence_before();
        __syncthreads();
        if (tid == 0) {
            fence_after();
            const uint32_t vaddr = s_base + kSmemV + (j & 1) * kTileBytes;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t poff = (ks >> 2) * (128 * 128) + (ks & 3) * 32;
                mma_f16(tmem + 256, sdesc(s_base + kSmemP + poff, 16, 1024),
                        sdesc(vaddr + ks * 16 * 128, 128 * 128, 1024), id_o, (j > 0 || ks > 0) ? 1u : 0u);
            }
            mma_commit(smem_u32(bars + 2));
        }
    }
    // last P.V
    if (ok && n_tiles > 0) {
        ok = __syncthreads_and(bar_wait(smem_u32(bars + 2), (n_tiles - 1) & 1)) != 0;
        fence_after();
    }
    if (!ok) {
        if (tid == 0) record_error(p.err, -3000);
    } else {
        s_red[hc * kRows + row] = l_part;
        __syncthreads();
        const float l_row = l_part + s_red[(hc ^ 1) * kRows + row];
        const float inv = l_row > 0.f ? 1.f / l_row : 0.f;
        // every thread reads its lane (tcgen05.ld is warp-collective); rows past
        // the request are not stored
        const int pos = R / G, hh = R - (R / G) * G;
        bf16 *orow = static_cast<bf16 *>(p.o) +
                     ((static_cast<int64_t>(qo0) + pos) * p.n_heads + g * G + hh) * kD + hc * 64;
        float ov[64];
        tmem_ld64(tO, ov);
#pragma unroll
        for (int c0 = 0; c0 < 64; c0 += 32) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
                __nv_bfloat162 h = __floats2bfloat162_rn(ov[c0 + i] * inv, ov[c0 + i + 1] * inv);
                pk[i >> 1] = *reinterpret_cast<uint32_t *>(&h);
            }
            if (R < rows) {
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4)
                    *reinterpret_cast<uint4 *>(orow + c0 + q4 * 8) =
                        make_uint4(pk[4 * q4], pk[4 * q4 + 1], pk[4 * q4 + 2], pk[4 * q4 + 3]);
            }
        }
    }
    cp_async_wait<0>();
    fence_before();
    __syncthreads();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(kTmemCols));
}

template <int G>
cudaError_t run(const PrefillParams &p, cudaStream_t s) {
    static std::atomic<uint64_t> attr_done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(attr_done.load() & bit)) {
        e = cudaFuncSetAttribute(prefill_tc_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_done.fetch_or(bit);
    }
    const int qtiles = (p.max_q_len * G + kRows - 1) / kRows;
    dim3 grid(qtiles, p.n_kv_heads, p.batch);
    prefill_tc_kernel<G><<<grid, kNT, kSmemBytes, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

bool prefill_tc_supported(int dtype, int head_dim, int group) {
    return dtype == PKV_BF16 && head_dim == 128 && (group == 1 || group == 2 || group == 4 || group == 8);
}

cudaError_t launch_prefill_tc(const PrefillParams &p, int group, cudaStream_t s) {
    switch (group) {
        case 1: return run<1>(p, s);
        case 2: return run<2>(p, s);
        case 4: return run<4>(p, s);
        case 8: return run<8>(p, s);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace pkv
