// pkv_decode_mma.cu -- bf16 paged decode on tensor cores (split pass).
//
// Same operation and workspace contract as the split kernel in
// pkv_decode.cu (AstrAI docs/guides/inference.md, "KV Cache" formula read
// through req_to_token, "Attention Backend" decode path); this is the bf16
// path.  The G query heads that share a kv head make the score block a real
// matrix product, so both products run as mma.sync m16n8k16 (bf16 in, fp32
// accumulate) with the heads as the N = 8 dimension:
//   S^T[16 tokens x 8 heads]  = K[16 x D] . Q^T[D x 8]       (A = K from smem)
//   O^T[D x 8 heads]         += V^T[D x 16] . P^T[16 x 8]     (A = V^T via ldmatrix.trans)
// P^T goes from the accumulator layout to the B-operand layout with two
// movmatrix transposes, so probabilities never touch shared memory.
//
// Two kernels share these building blocks:
//  - decode_mma_kernel: one CTA per (split, kv head, entry), four warps each
//    running its own cp.async ring over interleaved 16-token blocks (rows
//    XOR-swizzled in shared memory); used when n_kv_heads does not divide 8;
//  - decode_mma_allheads_kernel: one CTA reads whole slot rows of all kv
//    heads (K rows by bulk copy, V rows by cp.async, rows padded by 16 bytes
//    so ldmatrix is free of bank conflicts), either per (split, entry) or
//    over an exactly balanced partition of all tokens of the batch.  With 8
//    kv heads a CTA stages the slots of all its pieces at once and streams
//    them through one ring (stream_pieces); otherwise piece by piece.
// Slots come from req_to_token, or from a page table (slot_at).  The merge of
// the balanced partition (decode_merge_balanced_kernel) is at the end.
//
// Shared prefix (the caller states that the first shared_len positions of
// every row hold the same slots, as when prefix-cache hits give several
// requests the same pages): a separate instantiation of the all-heads kernel
// splits its CTAs into a group role (stream_group: the prefix read once per
// group of 16 / G requests, whose heads are the 16 columns of two n8 tiles,
// block_math2) and a private role (the balanced pass over the positions
// past the prefix); decode_merge_shared_kernel merges both kinds of pieces.
#include <atomic>

#include "pkv_common.cuh"
#include "pkv_launch.h"

namespace pkv {
namespace {

constexpr int kWarps = 4;
constexpr int kNT = kWarps * 32;
constexpr int kBlk = 16;          // tokens per block (the mma M / K extent)

template <int D>
struct MmaCfg {
    static constexpr int kStages = 3;
    static constexpr int kChunks = D / 8;                        // 16-byte chunks per row
    static constexpr int kBlkElems = kBlk * D;                   // one K (or V) block
    static constexpr int kStageElems = 2 * kBlkElems;            // K + V
    static constexpr size_t kSlotBytes = kDecodeMaxChunk * 4;
    static constexpr size_t kRingBytes = static_cast<size_t>(kWarps) * kStages * kStageElems * 2;
    static constexpr size_t kSmem = kSlotBytes + kRingBytes;
    static constexpr int kCpPerLane = 2 * kBlk * kChunks / 32;   // cp.async per lane per block
};

__device__ __forceinline__ int swz(int row, int chunk, int d) {
    return row * d + ((chunk ^ (row & 7)) << 3);
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void *p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void *p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(p)));
}
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(y) : "r"(x));
    return y;
}
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes)
                 : "memory");
}
// Bounded wait for the phase with the given parity.  Gives up after 2^18
// polls (each poll itself waits a short hardware-defined time) and returns
// false; the caller then records an error and stops waiting instead of
// hanging.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    for (int i = 0; i < (1 << 18); ++i) {
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

// Wait for the grid this one depends on programmatically (the cache write
// of a decode step) to complete and its writes to become visible.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }

// One bulk (TMA) copy of `bytes` contiguous bytes global -> shared, counted
// on the mbarrier `bar`.  Addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

template <int D, int G>
__global__ void __launch_bounds__(kNT, 2) decode_mma_kernel(const DecodeParams p) {
    using C = MmaCfg<D>;
    using bf16 = __nv_bfloat16;
    extern __shared__ __align__(128) unsigned char smem[];
    int *slots = reinterpret_cast<int *>(smem);
    bf16 *ring_all = reinterpret_cast<bf16 *>(smem + C::kSlotBytes);

    const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    int r = __ldg(p.req_pool_indices + b);
    if (static_cast<unsigned>(r) >= static_cast<unsigned>(p.num_reqs)) {
        record_error(p.err, r);
        r = 0;
    }
    int n = __ldg(p.seq_lens + b);
    const int n_cap = min(p.max_len, p.max_ctx_len);
    if (n < 0 || n > n_cap) {
        record_error(p.err, n);
        n = max(0, min(n, n_cap));
    }
    const int start = split * p.chunk;
    if (start >= n) {
        if (p.direct && n == 0) {
            bf16 *o = static_cast<bf16 *>(p.o) + (static_cast<int64_t>(b) * p.n_heads + g * G) * D;
            for (int i = tid; i < G * D; i += kNT) o[i] = __float2bfloat16_rn(0.f);
        }
        return;
    }
    const int len = min(p.chunk, n - start);

    const int32_t *row = p.req_to_token + static_cast<int64_t>(r) * p.max_ctx_len + start;
    for (int j = tid; j < len; j += kNT) {
        int sl = __ldg(row + j);
        if (static_cast<unsigned long long>(static_cast<long long>(sl)) >=
            static_cast<unsigned long long>(p.size)) {
            record_error(p.err, sl);
            sl = 0;
        }
        slots[j] = sl;
    }

    // Q^T B-fragments: lane holds head lane/4, dims ks*16 + 2*(lane%4) + {0,1} (+8)
    uint32_t qb[D / 16][2];
    {
        const int h = lane >> 2;
        const bf16 *qrow = static_cast<const bf16 *>(p.q) +
                           (static_cast<int64_t>(b) * p.n_heads + g * G + (h < G ? h : 0)) * D +
                           2 * (lane & 3);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            qb[ks][0] = h < G ? *reinterpret_cast<const uint32_t *>(qrow + ks * 16) : 0u;
            qb[ks][1] = h < G ? *reinterpret_cast<const uint32_t *>(qrow + ks * 16 + 8) : 0u;
        }
    }
    __syncthreads();

    const int64_t slot_stride = static_cast<int64_t>(p.n_kv_heads) * D;
    const bf16 *kbase = static_cast<const bf16 *>(p.k_buffer) + (p.layer_row0 * p.n_kv_heads + g) * D;
    const bf16 *vbase = static_cast<const bf16 *>(p.v_buffer) + (p.layer_row0 * p.n_kv_heads + g) * D;
    bf16 *ring = ring_all + static_cast<size_t>(warp) * C::kStages * C::kStageElems;

    const int nblk = (len + kBlk - 1) / kBlk;
    const int cnt = nblk > warp ? (nblk - warp + kWarps - 1) / kWarps : 0;

    // issue the copies of this warp's k-th block into ring stage `st`
    auto issue = [&](int k, int st) {
        const int t0 = (warp + k * kWarps) * kBlk;
        bf16 *dst0 = ring + st * C::kStageElems;
#pragma unroll
        for (int i = 0; i < C::kCpPerLane; ++i) {
            const int idx = lane + 32 * i;
            const int kv = idx / (kBlk * C::kChunks);
            const int rem = idx - kv * (kBlk * C::kChunks);
            const int t = rem / C::kChunks;
            const int c = rem - t * C::kChunks;
            bf16 *dst = dst0 + kv * C::kBlkElems + swz(t, c, D);
            const int tok = t0 + t;
            if (tok < len) {
                cp_async16(dst, (kv ? vbase : kbase) + slots[tok] * slot_stride + c * 8);
            } else {
                cp_async16(dst, kbase, 0);
            }
        }
    };

#pragma unroll
    for (int st = 0; st < C::kStages - 1; ++st) {
        if (st < cnt) issue(st, st);
        cp_async_commit();
    }

    float o_acc[D / 16][4];
#pragma unroll
    for (int i = 0; i < D / 16; ++i) o_acc[i][0] = o_acc[i][1] = o_acc[i][2] = o_acc[i][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY;   // running max, heads 2*(lane%4) and +1
    float l0 = 0.f, l1 = 0.f;               // lane-partial denominators

    for (int k = 0; k < cnt; ++k) {
        cp_async_wait<C::kStages - 2>();
        __syncwarp();
        if (k + C::kStages - 1 < cnt) issue(k + C::kStages - 1, (k + C::kStages - 1) % C::kStages);
        cp_async_commit();

        const bf16 *kt = ring + (k % C::kStages) * C::kStageElems;
        const bf16 *vt = kt + C::kBlkElems;
        const int valid = len - (warp + k * kWarps) * kBlk;   // >= 1

        // S^T = K Q^T
        float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            uint32_t a[4];
            ldsm_x4(a, kt + swz(lane & 15, 2 * ks + (lane >> 4), D));
            mma16816(s, a, qb[ks][0], qb[ks][1]);
        }
        const int tA = lane >> 2, tB = tA + 8;
        s[0] = tA < valid ? s[0] * p.scale_log2 : -INFINITY;
        s[1] = tA < valid ? s[1] * p.scale_log2 : -INFINITY;
        s[2] = tB < valid ? s[2] * p.scale_log2 : -INFINITY;
        s[3] = tB < valid ? s[3] * p.scale_log2 : -INFINITY;
        float mx0 = fmaxf(s[0], s[2]), mx1 = fmaxf(s[1], s[3]);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        const float al0 = exp2f(m0 - mn0), al1 = exp2f(m1 - mn1);
        m0 = mn0;
        m1 = mn1;
        const float p0 = exp2f(s[0] - mn0), p1 = exp2f(s[1] - mn1);
        const float p2 = exp2f(s[2] - mn0), p3 = exp2f(s[3] - mn1);
        l0 = l0 * al0 + p0 + p2;
        l1 = l1 * al1 + p1 + p3;
        if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
            for (int i = 0; i < D / 16; ++i) {
                o_acc[i][0] *= al0;
                o_acc[i][1] *= al1;
                o_acc[i][2] *= al0;
                o_acc[i][3] *= al1;
            }
        }
        // P^T (tokens x heads) -> B fragments (k = tokens, n = heads)
        const uint32_t pb0 = movmatrix_t(pack_bf16(p0, p1));
        const uint32_t pb1 = movmatrix_t(pack_bf16(p2, p3));
        // O^T += V^T P^T
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
            uint32_t a[4];
            ldsm_x4_t(a, vt + swz((lane & 7) + ((lane >> 4) << 3), 2 * mt + ((lane >> 3) & 1), D));
            mma16816(o_acc[mt], a, pb0, pb1);
        }
    }
    cp_async_wait<0>();

    // denominators: sum the lane partials over the 8 lanes sharing a head pair
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, off);
        l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }

    // combine the warps: red_o[w][h][D], red_ml[w][h][2]
    __syncthreads();
    float *red_o = reinterpret_cast<float *>(ring_all);
    float *red_ml = red_o + kWarps * G * D;
    const int h0 = 2 * (lane & 3), h1 = h0 + 1;
    if (lane < 4) {
        if (h0 < G) {
            red_ml[(warp * G + h0) * 2] = m0;
            red_ml[(warp * G + h0) * 2 + 1] = l0;
        }
        if (h1 < G) {
            red_ml[(warp * G + h1) * 2] = m1;
            red_ml[(warp * G + h1) * 2 + 1] = l1;
        }
    }
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
        const int d0 = mt * 16 + (lane >> 2);
        if (h0 < G) {
            red_o[(warp * G + h0) * D + d0] = o_acc[mt][0];
            red_o[(warp * G + h0) * D + d0 + 8] = o_acc[mt][2];
        }
        if (h1 < G) {
            red_o[(warp * G + h1) * D + d0] = o_acc[mt][1];
            red_o[(warp * G + h1) * D + d0 + 8] = o_acc[mt][3];
        }
    }
    __syncthreads();

    const int64_t bh0 = static_cast<int64_t>(b) * p.n_heads + g * G;
    for (int i = tid; i < G * D; i += kNT) {
        const int h = i / D, e = i - (i / D) * D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, red_ml[(w * G + h) * 2]);
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float sc = exp2f(red_ml[(w * G + h) * 2] - M);
            L += red_ml[(w * G + h) * 2 + 1] * sc;
            O += red_o[(w * G + h) * D + e] * sc;
        }
        const float out = O / L;
        if (p.direct) {
            static_cast<bf16 *>(p.o)[(bh0 + h) * D + e] = __float2bfloat16_rn(out);
        } else {
            const int64_t ps = (bh0 + h) * p.n_splits + split;
            p.o_part[ps * D + e] = out;
            if (e == 0) {
                p.ml_part[ps * 2] = M;
                p.ml_part[ps * 2 + 1] = L;
            }
        }
    }
}

// All kv heads in one CTA.  A stage holds TS = 128 / HK tokens of every kv
// head, so each slot's K (and V) row of n_kv_heads * D elements is fetched as
// one contiguous run (2 KB for 8 heads of 128 bf16) rather than as a 256-byte
// slice per CTA.  Warp w owns kv head w % HK and the 16-token block w / HK of
// each stage; warps that share a head are combined at the end of a segment.
//
// Two ways to hand out work:
//  - chunked: CTA (split, entry) takes tokens [split*chunk, (split+1)*chunk)
//    of one entry;
//  - balanced: the grid is n_parts CTAs over the flattened token space
//    [0, T), T = kv_indptr[batch]; CTA c takes [T*c/P, T*(c+1)/P) with
//    P = min(n_parts, T), walking across entries.  Its piece of entry b goes
//    to partial row (c + b) (rows are unique because pieces are ordered), or
//    straight to o when the piece is the whole entry.
template <int D, int HK>
struct AllHeadsCfg {
    static constexpr int kWarpsAH = 8;
    static constexpr int kNTAH = kWarpsAH * 32;
    static constexpr int kTS = kBlk * (kWarpsAH / HK);              // tokens per stage
    static constexpr int kRowElems = HK * D;                        // one slot row, all heads
    static constexpr int kRowBytes = kRowElems * 2;
    static constexpr int kPitch = kRowElems + 8;                    // +16 B: ldmatrix rows hit distinct banks
    static constexpr int kPartElems = kTS * kPitch;                 // the K (or V) part of a stage
    static constexpr int kStageElems = 2 * kPartElems;
    static constexpr size_t kStageBytes = static_cast<size_t>(kStageElems) * 2;
    static constexpr int kStages = 3;
    static constexpr size_t kSlotBytes = kDecodeMaxChunk * 4;
    static constexpr size_t kBarBytes = 64;
    static constexpr size_t kSmem = kSlotBytes + kBarBytes + kStages * kStageBytes;
    static_assert(kWarpsAH % HK == 0, "HK must divide 8");
    static_assert(kStageBytes % 16 == 0 && kRowBytes % 16 == 0, "bulk copies move 16-byte units");
};

// 2^x by the hardware approximation (ex2.approx.ftz: one instruction;
// results below 2^-126 flush to 0, 2^-inf = 0).  The softmax's weights are
// then rounded to bf16, far coarser than its error.
__device__ __forceinline__ float ex2_fast(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}

// One 16-token block of one kv head: scores S^T = K Q^T (16 tokens x 8
// heads), base-2 online softmax over the `valid` leading tokens (the rest
// score -inf), O^T += V^T P^T.  kt / vt point at the block's first row in
// shared memory (row pitch `pitch` elements).  m*/l* are the running max
// and sum of the two heads (columns) this lane holds.
template <int D>
__device__ __forceinline__ void block_math(const __nv_bfloat16 *kt, const __nv_bfloat16 *vt,
                                           int pitch, int valid, int lane, float scale_log2,
                                           const uint32_t (&qb)[D / 16][2], float (&o_acc)[D / 16][4],
                                           float &m0, float &m1, float &l0, float &l1) {
    float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
        uint32_t a[4];
        ldsm_x4(a, kt + (lane & 15) * pitch + (2 * ks + (lane >> 4)) * 8);
        mma16816(s, a, qb[ks][0], qb[ks][1]);
    }
    const int tA = lane >> 2, tB = tA + 8;
    s[0] = tA < valid ? s[0] * scale_log2 : -INFINITY;
    s[1] = tA < valid ? s[1] * scale_log2 : -INFINITY;
    s[2] = tB < valid ? s[2] * scale_log2 : -INFINITY;
    s[3] = tB < valid ? s[3] * scale_log2 : -INFINITY;
    float mx0 = fmaxf(s[0], s[2]), mx1 = fmaxf(s[1], s[3]);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float al0 = ex2_fast(m0 - mn0), al1 = ex2_fast(m1 - mn1);
    m0 = mn0;
    m1 = mn1;
    const float p0 = ex2_fast(s[0] - mn0), p1 = ex2_fast(s[1] - mn1);
    const float p2 = ex2_fast(s[2] - mn0), p3 = ex2_fast(s[3] - mn1);
    l0 = l0 * al0 + p0 + p2;
    l1 = l1 * al1 + p1 + p3;
    if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
        for (int i = 0; i < D / 16; ++i) {
            o_acc[i][0] *= al0;
            o_acc[i][1] *= al1;
            o_acc[i][2] *= al0;
            o_acc[i][3] *= al1;
        }
    }
    const uint32_t pb0 = movmatrix_t(pack_bf16(p0, p1));
    const uint32_t pb1 = movmatrix_t(pack_bf16(p2, p3));
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
        uint32_t a[4];
        ldsm_x4_t(a, vt + ((lane & 7) + ((lane >> 4) << 3)) * pitch + (2 * mt + ((lane >> 3) & 1)) * 8);
        mma16816(o_acc[mt], a, pb0, pb1);
    }
}

// Slot of position j of request row r: through req_to_token, or through the
// page table when p.page_size > 0.  A slot or page outside the pool is
// recorded and replaced by 0.
__device__ __forceinline__ int slot_at(const DecodeParams &p, int r, int j) {
    if (p.page_size > 0) {
        const int pg = __ldg(p.req_to_page + static_cast<int64_t>(r) * p.max_pages + j / p.page_size);
        if (static_cast<unsigned long long>(static_cast<long long>(pg)) >=
            static_cast<unsigned long long>(p.n_pages)) {
            record_error(p.err, pg);
            return 0;
        }
        return pg * p.page_size + j % p.page_size;
    }
    int sl = __ldg(p.req_to_token + static_cast<int64_t>(r) * p.max_ctx_len + j);
    if (static_cast<unsigned long long>(static_cast<long long>(sl)) >= static_cast<unsigned long long>(p.size)) {
        record_error(p.err, sl);
        sl = 0;
    }
    return sl;
}

// First CTA index of the balanced partition whose range holds token t.
__device__ __forceinline__ int part_of(long long t, long long T, int P) {
    const long long c = ((t + 1) * P - 1) / T;
    return static_cast<int>(c < P - 1 ? c : P - 1);
}

// Shared-prefix mode: the n_parts CTAs divide into the group role (p_sh CTAs
// over the group space [0, n_groups * shared_len)) and the private role (the
// rest, over the private space [0, T - batch * shared_len)) in proportion to
// the two token counts (group tokens weighted 9/8), with at least ceil(group space / 1024) group CTAs so
// that none stages more than 1024 positions.  The split and merge kernels
// derive it alike from T = kv_indptr[batch]; *_e are the CTAs that hold
// tokens (a role with fewer tokens than CTAs leaves the rest idle).
struct SharedRoles {
    long long t_sh, t_pr;
    int p_sh, p_pr, p_sh_e, p_pr_e;
};
__device__ __forceinline__ SharedRoles shared_roles(const DecodeParams &p, long long T) {
    SharedRoles r;
    r.t_sh = static_cast<long long>(p.n_groups) * p.shared_len;
    r.t_pr = T - static_cast<long long>(p.batch) * p.shared_len;
    const int P = p.n_parts;
    if (p.group_tc) {   // the group role is a kernel of its own
        r.t_sh = 0;
        r.p_sh = 0;
        r.p_pr = P;
    } else if (r.t_pr <= 0) {
        r.p_sh = P;
        r.p_pr = 0;
    } else {
        // a group token costs ~9/8 of a private one (16 query columns, not 8)
        const long long w_sh = 9 * r.t_sh, tot = w_sh + 8 * r.t_pr;
        long long psh = (static_cast<long long>(P) * w_sh + tot / 2) / tot;
        psh = max(psh, (r.t_sh + 1023) / 1024);
        psh = min(psh, static_cast<long long>(P - 1));
        r.p_sh = static_cast<int>(psh);
        r.p_pr = P - r.p_sh;
    }
    r.p_sh_e = static_cast<int>(min(static_cast<long long>(r.p_sh), r.t_sh));
    r.p_pr_e = r.t_pr > 0 ? static_cast<int>(min(static_cast<long long>(r.p_pr), r.t_pr)) : 0;
    return r;
}

// The raw table entry behind position j of request row r (the page id, or
// the slot with req_to_token); two rows share position j's slot iff these
// are equal.
__device__ __forceinline__ int table_entry(const DecodeParams &p, int r, int j) {
    if (p.page_size > 0)
        return __ldg(p.req_to_page + static_cast<int64_t>(r) * p.max_pages + j / p.page_size);
    return __ldg(p.req_to_token + static_cast<int64_t>(r) * p.max_ctx_len + j);
}

// block_math over two 8-column tiles of the score block (16 query columns):
// each K and V^T fragment is loaded from shared memory once and used by both
// tiles.  m / l hold, per tile, the running max and sum of this lane's two
// columns.
template <int D>
__device__ __forceinline__ void block_math2(const __nv_bfloat16 *kt, const __nv_bfloat16 *vt,
                                            int pitch, int valid, int lane, float scale_log2,
                                            const uint32_t (&qb)[2][D / 16][2],
                                            float (&o_acc)[2][D / 16][4], float (&m)[2][2],
                                            float (&l)[2][2]) {
    float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
        uint32_t a[4];
        ldsm_x4(a, kt + (lane & 15) * pitch + (2 * ks + (lane >> 4)) * 8);
        mma16816(s[0], a, qb[0][ks][0], qb[0][ks][1]);
        mma16816(s[1], a, qb[1][ks][0], qb[1][ks][1]);
    }
    const int tA = lane >> 2, tB = tA + 8;
    uint32_t pb[2][2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        s[t][0] = tA < valid ? s[t][0] * scale_log2 : -INFINITY;
        s[t][1] = tA < valid ? s[t][1] * scale_log2 : -INFINITY;
        s[t][2] = tB < valid ? s[t][2] * scale_log2 : -INFINITY;
        s[t][3] = tB < valid ? s[t][3] * scale_log2 : -INFINITY;
        float mx0 = fmaxf(s[t][0], s[t][2]), mx1 = fmaxf(s[t][1], s[t][3]);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        const float mn0 = fmaxf(m[t][0], mx0), mn1 = fmaxf(m[t][1], mx1);
        const float al0 = ex2_fast(m[t][0] - mn0), al1 = ex2_fast(m[t][1] - mn1);
        m[t][0] = mn0;
        m[t][1] = mn1;
        const float p0 = ex2_fast(s[t][0] - mn0), p1 = ex2_fast(s[t][1] - mn1);
        const float p2 = ex2_fast(s[t][2] - mn0), p3 = ex2_fast(s[t][3] - mn1);
        l[t][0] = l[t][0] * al0 + p0 + p2;
        l[t][1] = l[t][1] * al1 + p1 + p3;
        if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
            for (int i = 0; i < D / 16; ++i) {
                o_acc[t][i][0] *= al0;
                o_acc[t][i][1] *= al1;
                o_acc[t][i][2] *= al0;
                o_acc[t][i][3] *= al1;
            }
        }
        pb[t][0] = movmatrix_t(pack_bf16(p0, p1));
        pb[t][1] = movmatrix_t(pack_bf16(p2, p3));
    }
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
        uint32_t a[4];
        ldsm_x4_t(a, vt + ((lane & 7) + ((lane >> 4) << 3)) * pitch + (2 * mt + ((lane >> 3) & 1)) * 8);
        mma16816(o_acc[0][mt], a, pb[0][0], pb[0][1]);
        mma16816(o_acc[1][mt], a, pb[1][0], pb[1][1]);
    }
}

// Balanced-mode CTA c with one warp per kv head (8 kv heads), when its range
// [t0, t1) holds at most kMaxPieces entry pieces and their slots fit the slot
// array after rounding each piece up to whole 16-token stages.  Then:
//  - the pieces come from the metadata the caller read in one round trip
//    (ip: kv_indptr[KPT i .. KPT i + KPT], rq / sq: req_pool_indices /
//    seq_lens of this thread's KPT entries) and a block-wide scan;
//  - all slot indices are staged at once, each piece padded to a multiple
//    of 16 by repeating its last slot, so stage k is simply slots
//    [16k, 16k + 16) and the copy ring runs across piece boundaries without
//    draining;
//  - each warp finishes a piece straight from its registers (it owns its kv
//    head, so no cross-warp combine): o for a whole entry, else the partial
//    row (c + b).
// Returns false (having done nothing but read) when the range does not
// fit; the caller then takes the piece-by-piece path.
constexpr int kMaxPieces = 64;

template <int D, int G, int KPT>
__device__ __forceinline__ bool stream_pieces(const DecodeParams &p, int c, long long t0, long long t1,
                                              int n_cap, const int (&ip)[KPT + 1], const int (&rq)[KPT],
                                              const int (&sq)[KPT], int *slots, uint64_t *bars,
                                              __nv_bfloat16 *ring) {
    using C = AllHeadsCfg<D, 8>;
    using bf16 = __nv_bfloat16;
    constexpr int NW = C::kWarpsAH, NT = C::kNTAH, S = C::kStages;
    static_assert(C::kTS == 16, "one 16-token block per warp and stage");
    __shared__ int s_scan[NW][2];
    __shared__ int s_b[kMaxPieces], s_r[kMaxPieces], s_s0[kMaxPieces], s_len[kMaxPieces],
        s_off[kMaxPieces], s_direct[kMaxPieces];
    __shared__ int s_abort;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int e0 = tid * KPT;

    // this thread's pieces: non-empty, valid entries overlapping [t0, t1)
    int cnt = 0, pad = 0;
#pragma unroll
    for (int k = 0; k < KPT; ++k) {
        const long long lo = ip[k], hi = ip[k + 1];
        if (e0 + k < p.batch && hi > t0 && lo < t1 && hi > lo) {
            const bool ok = hi - lo == sq[k] && hi - lo <= n_cap && lo >= 0 &&
                            static_cast<unsigned>(rq[k]) < static_cast<unsigned>(p.num_reqs);
            if (ok) {
                ++cnt;
                pad += (static_cast<int>(min(hi, t1) - max(lo, t0)) + 15) & ~15;
            }
        }
    }
    // block-wide exclusive scan of (pieces, padded tokens) in entry order
    int ic = cnt, ipd = pad;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int a = __shfl_up_sync(0xffffffffu, ic, off), b = __shfl_up_sync(0xffffffffu, ipd, off);
        if (lane >= off) {
            ic += a;
            ipd += b;
        }
    }
    if (lane == 31) {
        s_scan[warp][0] = ic;
        s_scan[warp][1] = ipd;
    }
    if (tid == 0) s_abort = 0;
    __syncthreads();
    int n_pieces = 0, total = 0, cbase = ic - cnt, pbase = ipd - pad;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
        if (w < warp) {
            cbase += s_scan[w][0];
            pbase += s_scan[w][1];
        }
        n_pieces += s_scan[w][0];
        total += s_scan[w][1];
    }
    if (n_pieces > kMaxPieces || total > kDecodeMaxChunk) return false;   // CTA-uniform

    // the piece table, and errors for overlapping entries that fail validation
#pragma unroll
    for (int k = 0; k < KPT; ++k) {
        const long long lo = ip[k], hi = ip[k + 1];
        if (e0 + k < p.batch && hi > t0 && lo < t1 && hi > lo) {
            const bool ok = hi - lo == sq[k] && hi - lo <= n_cap && lo >= 0 &&
                            static_cast<unsigned>(rq[k]) < static_cast<unsigned>(p.num_reqs);
            if (!ok) {
                record_error(p.err, hi - lo);
                continue;
            }
            const int len = static_cast<int>(min(hi, t1) - max(lo, t0));
            s_b[cbase] = e0 + k;
            s_r[cbase] = rq[k];
            s_s0[cbase] = static_cast<int>(max(lo, t0) - lo);
            s_len[cbase] = len;
            s_off[cbase] = pbase;
            s_direct[cbase] = lo >= t0 && hi <= t1 && p.shared_len == 0;
            ++cbase;
            pbase += (len + 15) & ~15;
        }
    }
    __syncthreads();
    if (n_pieces == 0) return true;

    const int hw = warp;   // this warp's kv head
    // q of a piece for this warp: its G query heads of the piece's entry, G x D
    // bf16 contiguous in q (16-byte aligned).  Loaded a piece ahead with
    // 16-byte loads -- q may sit in host memory, where a few wide requests
    // cost far less than the mma fragment layout's 4-byte ones -- and turned
    // into fragments through this warp's slot of shared memory at the switch.
    constexpr int kQV = G * D / 8;         // 16-byte chunks per (piece, kv head)
    constexpr int kQL = (kQV + 31) / 32;   // per lane
    __shared__ __align__(16) uint4 s_q[NW][kQV];
    auto load_q = [&](int pc, uint4 (&qr)[kQL]) {
        const uint4 *src = reinterpret_cast<const uint4 *>(
            static_cast<const bf16 *>(p.q) + (static_cast<int64_t>(s_b[pc]) * p.n_heads + hw * G) * D);
#pragma unroll
        for (int j = 0; j < kQL; ++j)
            if (lane + 32 * j < kQV) qr[j] = src[lane + 32 * j];
    };
    auto to_frag = [&](const uint4 (&qr)[kQL], uint32_t (&qf)[D / 16][2]) {
        __syncwarp();   // every lane has read the previous piece's fragments
#pragma unroll
        for (int j = 0; j < kQL; ++j)
            if (lane + 32 * j < kQV) s_q[warp][lane + 32 * j] = qr[j];
        __syncwarp();
        const uint32_t *w = reinterpret_cast<const uint32_t *>(s_q[warp]);
        const int h = lane >> 2;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {   // columns 16 ks + 2 (lane % 4) and + 8 of head h
            qf[ks][0] = h < G ? w[h * (D / 2) + ks * 8 + (lane & 3)] : 0u;
            qf[ks][1] = h < G ? w[h * (D / 2) + ks * 8 + 4 + (lane & 3)] : 0u;
        }
    };
    uint4 q0[kQL], qn[kQL];   // the first and the next piece's q, in flight
    if (!p.q_staged) {   // a staged q is written by the cache write: read after the wait below
        load_q(0, q0);
        if (n_pieces > 1) load_q(1, qn);
    }

    // stage every slot index (padding rows repeat the piece's last slot)
    for (int j = tid; j < total; j += NT) {
        int a = 0, z = n_pieces - 1;   // last piece with s_off <= j
        while (a < z) {
            const int mid = (a + z + 1) >> 1;
            if (s_off[mid] <= j) a = mid; else z = mid - 1;
        }
        const int pos = min(j - s_off[a], s_len[a] - 1);
        slots[j] = slot_at(p, s_r[a], p.shared_len + s_s0[a] + pos);
    }
    __syncthreads();
    if (p.pdl) griddep_wait();   // K/V rows may come from the cache write before this kernel
    if (p.q_staged) {
        load_q(0, q0);
        if (n_pieces > 1) load_q(1, qn);
    }

    const int64_t slot_stride = static_cast<int64_t>(8) * D;
    const bf16 *kbase = static_cast<const bf16 *>(p.k_buffer) + p.layer_row0 * slot_stride;
    const bf16 *vbase = static_cast<const bf16 *>(p.v_buffer) + p.layer_row0 * slot_stride;
    const int nst = total / 16;
    // stage k: K rows by bulk copy (warp 0, one per token, on the stage's
    // mbarrier), V rows as 16-byte cp.async chunks from every thread (one
    // commit group per stage)
    auto issue = [&](int k) {
        const int st = k % S;
        bf16 *dst0 = ring + st * C::kStageElems;
        const int *sl = slots + k * 16;
        if (warp == 0) {
            const uint32_t bar = smem_u32(bars + st);
            if (lane == 0) mbar_expect_tx(bar, static_cast<uint32_t>(16 * C::kRowBytes));
            __syncwarp();
            if (lane < 16)
                bulk_g2s(smem_u32(dst0 + lane * C::kPitch), kbase + sl[lane] * slot_stride, C::kRowBytes, bar);
        }
        constexpr int kVChunks = C::kRowBytes / 16;
        bf16 *vdst = dst0 + C::kPartElems;
#pragma unroll
        for (int i = tid; i < 16 * kVChunks; i += NT) {
            const int t = i / kVChunks, ch = i - t * kVChunks;
            cp_async16(vdst + t * C::kPitch + ch * 8, vbase + sl[t] * slot_stride + ch * 8);
        }
        cp_async_commit();
    };
#pragma unroll
    for (int k = 0; k < S - 1; ++k) {
        if (k < nst) issue(k);
        else cp_async_commit();
    }

    uint32_t qb[D / 16][2];
    to_frag(q0, qb);   // its loads overlapped the slot staging
    float o_acc[D / 16][4];
#pragma unroll
    for (int i = 0; i < D / 16; ++i) o_acc[i][0] = o_acc[i][1] = o_acc[i][2] = o_acc[i][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    int pc = 0;                                        // piece being consumed
    int pend = (s_off[0] + ((s_len[0] + 15) & ~15)) >> 4;   // its end stage
    for (int k = 0; k < nst; ++k) {
        cp_async_wait<S - 2>();   // this thread's V chunks of stage k
        __syncthreads();          // stage k-1 is consumed; everyone's V of stage k landed
        if (s_abort) break;       // CTA-uniform after the barrier
        if (k + S - 1 < nst) issue(k + S - 1);
        else cp_async_commit();
        const bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(bars + k % S), (k / S) & 1));
        if (!ok) {
            if (lane == 0) {
                record_error(p.err, -1000 - k);
                s_abort = 1;
            }
            continue;
        }
        const bf16 *kt = ring + (k % S) * C::kStageElems + hw * D;
        block_math<D>(kt, kt + C::kPartElems, C::kPitch, s_len[pc] - (k * 16 - s_off[pc]), lane,
                      p.scale_log2, qb, o_acc, m0, m1, l0, l1);
        if (k + 1 < pend) continue;

        // piece pc is complete: normalise and write it from registers
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l0 += __shfl_xor_sync(0xffffffffu, l0, off);
            l1 += __shfl_xor_sync(0xffffffffu, l1, off);
        }
        const int b = s_b[pc];
        const int h0 = 2 * (lane & 3), h1 = h0 + 1;
        const float i0 = 1.f / l0, i1 = 1.f / l1;
        if (s_direct[pc]) {
            bf16 *o = static_cast<bf16 *>(p.o) + (static_cast<int64_t>(b) * p.n_heads + hw * G) * D;
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
                const int d = mt * 16 + (lane >> 2);
                if (h0 < G) {
                    o[h0 * D + d] = __float2bfloat16_rn(o_acc[mt][0] * i0);
                    o[h0 * D + d + 8] = __float2bfloat16_rn(o_acc[mt][2] * i0);
                }
                if (h1 < G) {
                    o[h1 * D + d] = __float2bfloat16_rn(o_acc[mt][1] * i1);
                    o[h1 * D + d + 8] = __float2bfloat16_rn(o_acc[mt][3] * i1);
                }
            }
        } else {
            const int64_t row = (static_cast<int64_t>(c) + b) * p.n_heads + hw * G;
            float *op = p.o_part + row * D;
            const uint64_t pol = l2_keep_policy();
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
                const int d = mt * 16 + (lane >> 2);
                if (h0 < G) {
                    st_keep(op + h0 * D + d, o_acc[mt][0] * i0, pol);
                    st_keep(op + h0 * D + d + 8, o_acc[mt][2] * i0, pol);
                }
                if (h1 < G) {
                    st_keep(op + h1 * D + d, o_acc[mt][1] * i1, pol);
                    st_keep(op + h1 * D + d + 8, o_acc[mt][3] * i1, pol);
                }
            }
            if (lane < 4) {
                if (h0 < G) {
                    st_keep(p.ml_part + (row + h0) * 2, m0, pol);
                    st_keep(p.ml_part + (row + h0) * 2 + 1, l0, pol);
                }
                if (h1 < G) {
                    st_keep(p.ml_part + (row + h1) * 2, m1, pol);
                    st_keep(p.ml_part + (row + h1) * 2 + 1, l1, pol);
                }
            }
        }
        if (++pc == n_pieces) break;
        pend = (s_off[pc] + ((s_len[pc] + 15) & ~15)) >> 4;
#pragma unroll
        for (int i = 0; i < D / 16; ++i) o_acc[i][0] = o_acc[i][1] = o_acc[i][2] = o_acc[i][3] = 0.f;
        to_frag(qn, qb);
        m0 = m1 = -INFINITY;
        l0 = l1 = 0.f;
        if (pc + 1 < n_pieces) load_q(pc + 1, qn);
    }
    cp_async_wait<0>();
    return true;
}

// Group role of the shared-prefix mode (one warp per kv head, 8 kv heads).
// CTA cs covers [t0, t1) of the group space, where group gi owns
// [gi * Ts, gi * Ts + Ts): the shared positions of entries gi * R ..
// gi * R + R - 1 (R = 16 / G).  Each group piece is read once for all its
// entries: column col = 8 t + (lane >> 2) of n-tile t is entry
// gi * R + col / G, head hw * G + col % G (columns past the batch hold
// q = 0 and are not written).  All slot indices are staged at once, from
// the group's first entry, each piece padded to whole 16-token stages; every
// other member's table entries over the piece are compared with the
// first's and a mismatch is recorded (the shared-prefix claim was false).
// Each piece ends in one partial per (member, head).
template <int D, int G>
__device__ __forceinline__ void stream_group(const DecodeParams &p, int cs, long long t0, long long t1,
                                             int *slots, uint64_t *bars, __nv_bfloat16 *ring) {
    using C = AllHeadsCfg<D, 8>;
    using bf16 = __nv_bfloat16;
    constexpr int NT = C::kNTAH, S = C::kStages, R = 16 / G;
    constexpr int kMaxGroupPieces = 24;
    static_assert(C::kTS == 16, "one 16-token block per warp and stage");
    __shared__ int g_gi[kMaxGroupPieces], g_s0[kMaxGroupPieces], g_len[kMaxGroupPieces],
        g_off[kMaxGroupPieces], g_r[kMaxGroupPieces];
    __shared__ int g_n, g_total, g_abort;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int Ts = p.shared_len;

    if (tid == 0) {
        int n = 0, off = 0;
        for (long long gi = t0 / Ts; gi * Ts < t1; ++gi) {
            const long long lo = gi * Ts;
            const int s0 = static_cast<int>(max(t0, lo) - lo);
            const int len = static_cast<int>(min(t1, lo + Ts) - lo) - s0;
            if (len <= 0) continue;
            if (n == kMaxGroupPieces || off + ((len + 15) & ~15) > kDecodeMaxChunk) {
                record_error(p.err, -200000 - cs);   // the host keeps ranges within these bounds
                break;
            }
            int r = __ldg(p.req_pool_indices + gi * R);
            if (static_cast<unsigned>(r) >= static_cast<unsigned>(p.num_reqs)) {
                record_error(p.err, r);
                r = 0;
            }
            g_gi[n] = static_cast<int>(gi);
            g_s0[n] = s0;
            g_len[n] = len;
            g_off[n] = off;
            g_r[n] = r;
            off += (len + 15) & ~15;
            ++n;
        }
        g_n = n;
        g_total = off;
        g_abort = 0;
    }
    __syncthreads();
    const int n_pieces = g_n, total = g_total;
    if (n_pieces == 0) return;

    const int hw = warp;   // this warp's kv head
    auto load_q = [&](int pc, uint32_t (&qr)[2][D / 16][2]) {
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            const int col = 8 * t + (lane >> 2);
            const int b = g_gi[pc] * R + col / G;
            const bool ok = b < p.batch;
            const bf16 *qrow = static_cast<const bf16 *>(p.q) +
                               (static_cast<int64_t>(ok ? b : 0) * p.n_heads + hw * G + col % G) * D +
                               2 * (lane & 3);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                qr[t][ks][0] = ok ? *reinterpret_cast<const uint32_t *>(qrow + ks * 16) : 0u;
                qr[t][ks][1] = ok ? *reinterpret_cast<const uint32_t *>(qrow + ks * 16 + 8) : 0u;
            }
        }
    };
    uint32_t qb[2][D / 16][2];
    load_q(0, qb);

    // stage every slot index (padding rows repeat the piece's last slot)
    for (int j = tid; j < total; j += NT) {
        int a = 0;
        while (a + 1 < n_pieces && g_off[a + 1] <= j) ++a;
        const int pos = min(j - g_off[a], g_len[a] - 1);
        slots[j] = slot_at(p, g_r[a], g_s0[a] + pos);
    }
    __syncthreads();
    if (p.pdl) griddep_wait();   // K/V rows may come from the cache write before this kernel

    const int64_t slot_stride = static_cast<int64_t>(8) * D;
    const bf16 *kbase = static_cast<const bf16 *>(p.k_buffer) + p.layer_row0 * slot_stride;
    const bf16 *vbase = static_cast<const bf16 *>(p.v_buffer) + p.layer_row0 * slot_stride;
    const int nst = total / 16;
    auto issue = [&](int k) {
        const int st = k % S;
        bf16 *dst0 = ring + st * C::kStageElems;
        const int *sl = slots + k * 16;
        if (warp == 0) {
            const uint32_t bar = smem_u32(bars + st);
            if (lane == 0) mbar_expect_tx(bar, static_cast<uint32_t>(16 * C::kRowBytes));
            __syncwarp();
            if (lane < 16)
                bulk_g2s(smem_u32(dst0 + lane * C::kPitch), kbase + sl[lane] * slot_stride, C::kRowBytes, bar);
        }
        constexpr int kVChunks = C::kRowBytes / 16;
        bf16 *vdst = dst0 + C::kPartElems;
#pragma unroll
        for (int i = tid; i < 16 * kVChunks; i += NT) {
            const int t = i / kVChunks, ch = i - t * kVChunks;
            cp_async16(vdst + t * C::kPitch + ch * 8, vbase + sl[t] * slot_stride + ch * 8);
        }
        cp_async_commit();
    };
#pragma unroll
    for (int k = 0; k < S - 1; ++k) {
        if (k < nst) issue(k);
        else cp_async_commit();
    }
    // with the first stages in flight: the other members' table entries must
    // equal the first member's wherever a new entry (page) starts
    for (int j = tid; j < total; j += NT) {
        int a = 0;
        while (a + 1 < n_pieces && g_off[a + 1] <= j) ++a;
        const int rel = j - g_off[a];
        const int jp = g_s0[a] + rel;
        if (rel >= g_len[a] || (p.page_size > 0 && jp % p.page_size != 0 && rel != 0)) continue;
        const int lead = table_entry(p, g_r[a], jp);
        for (int u = 1; u < R; ++u) {
            const int b = g_gi[a] * R + u;
            if (b >= p.batch) break;
            const int r = __ldg(p.req_pool_indices + b);
            if (static_cast<unsigned>(r) >= static_cast<unsigned>(p.num_reqs)) {
                record_error(p.err, r);
                continue;
            }
            if (table_entry(p, r, jp) != lead) record_error(p.err, -100000 - b);
        }
    }

    float o_acc[2][D / 16][4];
    float m[2][2], l[2][2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
#pragma unroll
        for (int i = 0; i < D / 16; ++i) o_acc[t][i][0] = o_acc[t][i][1] = o_acc[t][i][2] = o_acc[t][i][3] = 0.f;
        m[t][0] = m[t][1] = -INFINITY;
        l[t][0] = l[t][1] = 0.f;
    }
    int pc = 0;
    int pend = (g_off[0] + ((g_len[0] + 15) & ~15)) >> 4;
    for (int k = 0; k < nst; ++k) {
        cp_async_wait<S - 2>();
        __syncthreads();
        if (g_abort) break;   // CTA-uniform after the barrier
        if (k + S - 1 < nst) issue(k + S - 1);
        else cp_async_commit();
        const bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(bars + k % S), (k / S) & 1));
        if (!ok) {
            if (lane == 0) {
                record_error(p.err, -1000 - k);
                g_abort = 1;
            }
            continue;
        }
        const bf16 *kt = ring + (k % S) * C::kStageElems + hw * D;
        block_math2<D>(kt, kt + C::kPartElems, C::kPitch, g_len[pc] - (k * 16 - g_off[pc]), lane,
                       p.scale_log2, qb, o_acc, m, l);
        if (k + 1 < pend) continue;

        // piece pc is complete: one partial per (member, head) from registers
        const int gi = g_gi[pc];
#pragma unroll
        for (int t = 0; t < 2; ++t) {
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                l[t][0] += __shfl_xor_sync(0xffffffffu, l[t][0], off);
                l[t][1] += __shfl_xor_sync(0xffffffffu, l[t][1], off);
            }
#pragma unroll
            for (int x = 0; x < 2; ++x) {
                const int col = 8 * t + 2 * (lane & 3) + x;
                const int u = col / G;
                if (gi * R + u >= p.batch) continue;
                const int64_t unit = p.group_unit0 +
                                     (static_cast<int64_t>(cs + gi) * R + u) * p.n_heads + hw * G + col % G;
                float *op = p.o_part + unit * D;
                const float inv = 1.f / l[t][x];
                const uint64_t pol = l2_keep_policy();
#pragma unroll
                for (int mt = 0; mt < D / 16; ++mt) {
                    const int d = mt * 16 + (lane >> 2);
                    st_keep(op + d, o_acc[t][mt][x] * inv, pol);
                    st_keep(op + d + 8, o_acc[t][mt][2 + x] * inv, pol);
                }
                if (lane < 4) {
                    st_keep(p.ml_part + unit * 2, m[t][x], pol);
                    st_keep(p.ml_part + unit * 2 + 1, l[t][x], pol);
                }
            }
        }
        if (++pc == n_pieces) break;
        pend = (g_off[pc] + ((g_len[pc] + 15) & ~15)) >> 4;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
#pragma unroll
            for (int i = 0; i < D / 16; ++i)
                o_acc[t][i][0] = o_acc[t][i][1] = o_acc[t][i][2] = o_acc[t][i][3] = 0.f;
            m[t][0] = m[t][1] = -INFINITY;
            l[t][0] = l[t][1] = 0.f;
        }
        load_q(pc, qb);
    }
    cp_async_wait<0>();
}

// kShared: the shared-prefix mode's instantiation (both roles); the plain
// one holds no group-role code, so its register budget is its own.
template <int D, int G, int HK, bool kShared>
__global__ void __launch_bounds__(AllHeadsCfg<D, HK>::kNTAH, 1)
decode_mma_allheads_kernel(const DecodeParams p) {
    using C = AllHeadsCfg<D, HK>;
    using bf16 = __nv_bfloat16;
    constexpr int NW = C::kWarpsAH, NT = C::kNTAH;
    extern __shared__ __align__(128) unsigned char smem[];
    int *slots = reinterpret_cast<int *>(smem);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kSlotBytes);   // one per stage
    bf16 *ring = reinterpret_cast<bf16 *>(smem + C::kSlotBytes + C::kBarBytes);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // The merge kernel (launched as a programmatic dependent) may start its
    // prologue now; it waits for this grid's completion before reading partials.
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    if (tid == 0) {
        for (int st = 0; st < C::kStages; ++st) mbar_init(smem_u32(bars + st), 1);
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    __syncthreads();
    uint32_t issued = 0;               // stages issued by this CTA so far (phase bookkeeping)
    __shared__ int s_abort;            // set once a wait gave up: no further copies or waits
    if (tid == 0) s_abort = 0;
    const int hw = warp % HK;          // this warp's kv head
    const int blk = warp / HK;         // this warp's 16-token block within a stage
    const int n_cap = min(p.max_len, p.max_ctx_len);
    const int64_t slot_stride = static_cast<int64_t>(HK) * D;
    const bf16 *kbase = static_cast<const bf16 *>(p.k_buffer) + p.layer_row0 * slot_stride;
    const bf16 *vbase = static_cast<const bf16 *>(p.v_buffer) + p.layer_row0 * slot_stride;

    // Process positions [s0, s1) of entry b (request row r) and write the
    // result to o (direct) or to partial row `prow` (n_heads rows per index).
    auto segment = [&](int b, int r, int s0, int s1, bool direct, int64_t prow, int64_t pstride) {
        uint32_t qb[D / 16][2];
        {
            const int h = lane >> 2;
            const bf16 *qrow = static_cast<const bf16 *>(p.q) +
                               (static_cast<int64_t>(b) * p.n_heads + hw * G + (h < G ? h : 0)) * D +
                               2 * (lane & 3);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                qb[ks][0] = h < G ? *reinterpret_cast<const uint32_t *>(qrow + ks * 16) : 0u;
                qb[ks][1] = h < G ? *reinterpret_cast<const uint32_t *>(qrow + ks * 16 + 8) : 0u;
            }
        }
        float o_acc[D / 16][4];
#pragma unroll
        for (int i = 0; i < D / 16; ++i) o_acc[i][0] = o_acc[i][1] = o_acc[i][2] = o_acc[i][3] = 0.f;
        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
        for (int pc = s0; pc < s1; pc += kDecodeMaxChunk) {
            const int len = min(kDecodeMaxChunk, s1 - pc);
            for (int j = tid; j < len; j += NT) slots[j] = slot_at(p, r, pc + j);
            __syncthreads();
            const int nst = (len + C::kTS - 1) / C::kTS;
            const uint32_t first = issued;   // global index of this piece's stage 0
            // Stage k: the K rows go through the bulk-copy (TMA) engine, one
            // copy per token row of all kv heads, counted on the stage's
            // mbarrier (issued by warp 0); the V rows go through the load/store
            // path as 16-byte cp.async chunks from every thread, one commit
            // group per stage.  Splitting the bytes between the two copy
            // engines keeps either from capping the stream.  Rows past the
            // piece repeat the first token's row so the stage holds finite data.
            auto issue = [&](int k) {
                const uint32_t g = first + k;
                const int st = g % C::kStages;
                bf16 *dst0 = ring + st * C::kStageElems;
                if (warp == 0) {
                    const uint32_t bar = smem_u32(bars + st);
                    if (lane == 0) mbar_expect_tx(bar, static_cast<uint32_t>(C::kTS * C::kRowBytes));
                    __syncwarp();
                    for (int t = lane; t < C::kTS; t += 32) {
                        const int tok = k * C::kTS + t;
                        bulk_g2s(smem_u32(dst0 + t * C::kPitch),
                                 kbase + slots[tok < len ? tok : 0] * slot_stride, C::kRowBytes, bar);
                    }
                }
                constexpr int kVChunks = C::kRowBytes / 16;   // per token row
                bf16 *vdst = dst0 + C::kPartElems;
#pragma unroll
                for (int i = tid; i < C::kTS * kVChunks; i += NT) {
                    const int t = i / kVChunks, c = i - t * kVChunks;
                    const int tok = k * C::kTS + t;
                    cp_async16(vdst + t * C::kPitch + c * 8,
                               vbase + slots[tok < len ? tok : 0] * slot_stride + c * 8);
                }
                cp_async_commit();
            };
            if (!s_abort) {
                for (int k = 0; k < C::kStages - 1; ++k) {
                    if (k < nst) issue(k);
                    else cp_async_commit();
                }
            }
            issued += nst;
            for (int k = 0; k < nst; ++k) {
                cp_async_wait<C::kStages - 2>();   // this thread's V chunks of stage k
                __syncthreads();   // stage k-1 is consumed; everyone's V of stage k landed
                if (s_abort) continue;   // CTA-uniform after the barrier
                if (k + C::kStages - 1 < nst) issue(k + C::kStages - 1);
                else cp_async_commit();
                const uint32_t g = first + k;
                const bool ok = __all_sync(0xffffffffu,
                                           mbar_wait(smem_u32(bars + g % C::kStages), (g / C::kStages) & 1));
                if (!ok) {
                    if (lane == 0) {
                        record_error(p.err, -1000 - k);
                        s_abort = 1;
                    }
                    continue;
                }

                const int valid = len - (k * C::kTS + blk * kBlk);
                if (valid <= 0) continue;   // warp-uniform
                const bf16 *kt = ring + ((first + k) % C::kStages) * C::kStageElems +
                                 blk * kBlk * C::kPitch + hw * D;
                block_math<D>(kt, kt + C::kPartElems, C::kPitch, valid, lane, p.scale_log2, qb, o_acc,
                              m0, m1, l0, l1);
            }
            cp_async_wait<0>();
            __syncthreads();   // ring and slots are free for the next piece / the combine
        }

#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l0 += __shfl_xor_sync(0xffffffffu, l0, off);
            l1 += __shfl_xor_sync(0xffffffffu, l1, off);
        }
        float *red_o = reinterpret_cast<float *>(ring);   // [NW][G][D]
        float *red_ml = red_o + NW * G * D;               // [NW][G][2]
        const int h0 = 2 * (lane & 3), h1 = h0 + 1;
        if (lane < 4) {
            if (h0 < G) {
                red_ml[(warp * G + h0) * 2] = m0;
                red_ml[(warp * G + h0) * 2 + 1] = l0;
            }
            if (h1 < G) {
                red_ml[(warp * G + h1) * 2] = m1;
                red_ml[(warp * G + h1) * 2 + 1] = l1;
            }
        }
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
            const int d0 = mt * 16 + (lane >> 2);
            if (h0 < G) {
                red_o[(warp * G + h0) * D + d0] = o_acc[mt][0];
                red_o[(warp * G + h0) * D + d0 + 8] = o_acc[mt][2];
            }
            if (h1 < G) {
                red_o[(warp * G + h1) * D + d0] = o_acc[mt][1];
                red_o[(warp * G + h1) * D + d0 + 8] = o_acc[mt][3];
            }
        }
        __syncthreads();
        const int64_t bh0 = static_cast<int64_t>(b) * p.n_heads;
        for (int i = tid; i < HK * G * D; i += NT) {
            const int gh = i / D, e = i - gh * D;
            const int g = gh / G, h = gh - g * G;
            float M = -INFINITY;
#pragma unroll
            for (int w = g; w < NW; w += HK) M = fmaxf(M, red_ml[(w * G + h) * 2]);
            float L = 0.f, O = 0.f;
#pragma unroll
            for (int w = g; w < NW; w += HK) {
                const float sc = exp2f(red_ml[(w * G + h) * 2] - M);
                L += red_ml[(w * G + h) * 2 + 1] * sc;
                O += red_o[(w * G + h) * D + e] * sc;
            }
            const float out = O / L;
            if (direct) {
                static_cast<bf16 *>(p.o)[(bh0 + gh) * D + e] = __float2bfloat16_rn(out);
            } else {
                const int64_t ps = prow + gh * pstride;
                p.o_part[ps * D + e] = out;
                if (e == 0) {
                    p.ml_part[ps * 2] = M;
                    p.ml_part[ps * 2 + 1] = L;
                }
            }
        }
        // the combine area is the ring of the next segment, which the bulk
        // copies (async proxy) will overwrite
        asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
        __syncthreads();
    };

    if (!p.balanced) {
        if (p.pdl) griddep_wait();
        const int split = blockIdx.x, b = blockIdx.y;
        int r = __ldg(p.req_pool_indices + b);
        if (static_cast<unsigned>(r) >= static_cast<unsigned>(p.num_reqs)) {
            record_error(p.err, r);
            r = 0;
        }
        int n = __ldg(p.seq_lens + b);
        if (n < 0 || n > n_cap) {
            record_error(p.err, n);
            n = max(0, min(n, n_cap));
        }
        const int start = split * p.chunk;
        if (start >= n) {
            if (p.direct && n == 0) {
                bf16 *o = static_cast<bf16 *>(p.o) + static_cast<int64_t>(b) * p.n_heads * D;
                for (int i = tid; i < p.n_heads * D; i += NT) o[i] = __float2bfloat16_rn(0.f);
            }
            return;
        }
        segment(b, r, start, min(n, start + p.chunk), p.direct != 0,
                static_cast<int64_t>(b) * p.n_heads * p.n_splits + split, p.n_splits);
        return;
    }

    // balanced partition of [0, T)
    int c = blockIdx.x;
    // With one warp per kv head (HK == NW) and at most KPT * NT entries, the
    // entries' metadata comes in one round trip together with T: thread i
    // holds entries [KPT i, KPT i + KPT).
    constexpr int KPT = 4;
    constexpr bool kFast = HK == NW;
    const bool fast_batch = kFast && p.batch <= KPT * NT;
    const int e0 = tid * KPT;
    int ip[KPT + 1], rq[KPT], sq[KPT];
#pragma unroll
    for (int k = 0; k <= KPT; ++k) ip[k] = fast_batch && e0 + k <= p.batch ? __ldg(p.kv_indptr + e0 + k) : 0;
#pragma unroll
    for (int k = 0; k < KPT; ++k) {
        rq[k] = fast_batch && e0 + k < p.batch ? __ldg(p.req_pool_indices + e0 + k) : 0;
        sq[k] = fast_batch && e0 + k < p.batch ? __ldg(p.seq_lens + e0 + k) : 0;
    }
    const long long T = __ldg(p.kv_indptr + p.batch);
    if (T <= 0) return;
    // Shared-prefix mode (shared_len > 0; 8 kv heads): the first CTAs take
    // the group role; the others partition the private space, where entry b
    // holds [kv_indptr[b] - b Ts, kv_indptr[b + 1] - (b + 1) Ts) and offset
    // x stands for position Ts + x.  Ts = 0: the plain balanced partition.
    const long long Ts = kShared ? p.shared_len : 0;
    long long Tw = T;
    int P;
    if (kShared) {
        const SharedRoles ro = shared_roles(p, T);
        if (c < ro.p_sh) {
            if constexpr (kFast && kShared) {
                if (c < ro.p_sh_e)
                    stream_group<D, G>(p, c, ro.t_sh * c / ro.p_sh_e, ro.t_sh * (c + 1) / ro.p_sh_e, slots,
                                       bars, ring);
            }
            return;
        }
        c -= ro.p_sh;
        P = ro.p_pr_e;
        Tw = ro.t_pr;
#pragma unroll
        for (int k = 0; k <= KPT; ++k)
            if (e0 + k <= p.batch) ip[k] = static_cast<int>(ip[k] - (e0 + k) * Ts);
#pragma unroll
        for (int k = 0; k < KPT; ++k) {
            if (e0 + k < p.batch && fast_batch) {
                if (sq[k] < Ts) record_error(p.err, sq[k]);   // shorter than the shared prefix
                sq[k] = static_cast<int>(sq[k] - Ts);
            }
        }
    } else {
        P = static_cast<int>(min(static_cast<long long>(p.n_parts), T));
    }
    if (c >= P) return;
    const int n_cap_w = static_cast<int>(n_cap - Ts);   // longest private range
    long long t0 = Tw * c / P;
    const long long t1 = Tw * (c + 1) / P;

    if constexpr (kFast) {
        if (fast_batch && stream_pieces<D, G, KPT>(p, c, t0, t1, n_cap_w, ip, rq, sq, slots, bars, ring))
            return;
    }

    if (p.pdl) griddep_wait();   // piece-by-piece pass: wait before anything streams
    auto ipw = [&](int e) { return static_cast<long long>(__ldg(p.kv_indptr + e)) - e * Ts; };
    int lo_b = 0, hi_b = p.batch - 1;   // first entry whose range ends after t0
    while (lo_b < hi_b) {
        const int mid = (lo_b + hi_b) >> 1;
        if (ipw(mid + 1) > t0) hi_b = mid; else lo_b = mid + 1;
    }
    for (int b = lo_b; b < p.batch && t0 < t1; ++b) {
        const long long lo = ipw(b), hi = ipw(b + 1);
        if (hi <= t0) continue;
        const long long n = hi - lo;
        int r = __ldg(p.req_pool_indices + b);
        if (n != __ldg(p.seq_lens + b) - Ts || n > n_cap_w || lo < 0 ||
            static_cast<unsigned>(r) >= static_cast<unsigned>(p.num_reqs)) {
            record_error(p.err, n);
            t0 = hi;
            continue;
        }
        const int s0 = static_cast<int>(t0 - lo);
        const int s1 = static_cast<int>(min(t1, hi) - lo);
        const bool whole = s0 == 0 && s1 == n && Ts == 0;
        segment(b, r, static_cast<int>(s0 + Ts), static_cast<int>(s1 + Ts), whole,
                (static_cast<int64_t>(c) + b) * p.n_heads, 1);
        t0 = lo + s1;
    }
}

template <int D, int G, int HK, bool kShared>
cudaError_t run_allheads_k(const DecodeParams &p, cudaStream_t s) {
    using C = AllHeadsCfg<D, HK>;
    static std::atomic<uint64_t> attr_done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(attr_done.load() & bit)) {
        e = cudaFuncSetAttribute(decode_mma_allheads_kernel<D, G, HK, kShared>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(C::kSmem));
        if (e != cudaSuccess) return e;
        attr_done.fetch_or(bit);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = p.balanced ? dim3(p.n_parts, 1) : dim3(p.n_splits, p.batch);
    cfg.blockDim = dim3(C::kNTAH);
    cfg.dynamicSmemBytes = C::kSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = p.pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, decode_mma_allheads_kernel<D, G, HK, kShared>, p);
}

template <int D, int G, int HK>
cudaError_t run_allheads(const DecodeParams &p, cudaStream_t s) {
    if constexpr (HK == 8) {
        if (p.shared_len > 0) return run_allheads_k<D, G, HK, true>(p, s);
    }
    return run_allheads_k<D, G, HK, false>(p, s);
}

template <int D, int G>
cudaError_t run_hk(const DecodeParams &p, cudaStream_t s) {
    switch (p.n_kv_heads) {
        case 1: return run_allheads<D, G, 1>(p, s);
        case 2: return run_allheads<D, G, 2>(p, s);
        case 4: return run_allheads<D, G, 4>(p, s);
        case 8: return run_allheads<D, G, 8>(p, s);
        default: return cudaErrorNotSupported;
    }
}

// Merge of the balanced mode.  Entry b's pieces are partial rows c + b for c
// in [part_of(lo), part_of(hi - 1)] (a single piece was written to o by the
// split kernel).  WPI warps merge one (entry, head); warp `sub` takes pieces
// sub, sub + WPI, ... kBatch at a time, loading each piece's (m, l) (the
// same address in every lane) and its float4 columns together, so one
// round trip to L2 brings a whole batch.  A batch folds into the warp's
// running (M, L, acc) with one rescale; WPI > 1 warps then combine through
// shared memory.
template <int D, int WPI>
__global__ void __launch_bounds__(WPI > 8 ? 32 * WPI : 256) decode_merge_balanced_kernel(const DecodeParams p) {
    constexpr int NW = WPI > 8 ? WPI : 8, IPC = NW / WPI, kCols = D / 4;
    constexpr int kBatch = WPI == 16 ? 10 : 8;
    __shared__ float red_ml[NW][2];
    __shared__ float4 red_o[NW][kCols];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int grp = warp / WPI, sub = warp % WPI;
    const int item = blockIdx.x * IPC + grp;
    const int n_items = p.batch * p.n_heads;

    float M = -INFINITY, L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    bool merge = false;
    int64_t row0 = 0;
    __nv_bfloat16 *out = nullptr;
    if (item < n_items) {
        const int b = item / p.n_heads, h = item - b * p.n_heads;
        out = static_cast<__nv_bfloat16 *>(p.o) + static_cast<int64_t>(item) * D;
        const long long T = __ldg(p.kv_indptr + p.batch);
        const long long lo = __ldg(p.kv_indptr + b), hi = __ldg(p.kv_indptr + b + 1);
        const long long n = hi - lo;
        const int n_cap = min(p.max_len, p.max_ctx_len);
        const bool ok = T > 0 && n > 0 && n == __ldg(p.seq_lens + b) && n <= n_cap && lo >= 0 && hi <= T;
        if (!ok) {   // empty (or rejected) entry: o = 0
            asm volatile("griddepcontrol.wait;\n" ::: "memory");
            if (sub == 0)
                for (int e = lane; e < D; e += 32) out[e] = __float2bfloat16_rn(0.f);
        } else {
            const int P = static_cast<int>(min(static_cast<long long>(p.n_parts), T));
            const int c_lo = part_of(lo, T, P), c_hi = part_of(hi - 1, T, P);
            const int np = c_hi - c_lo + 1;
            merge = np > 1;   // one piece: written by the split kernel
            row0 = (static_cast<int64_t>(c_lo) + b) * p.n_heads + h;
            // the partials come from the split kernel, which may still run
            asm volatile("griddepcontrol.wait;\n" ::: "memory");
            if (merge) {
                const int mine = np > sub ? (np - sub + WPI - 1) / WPI : 0;   // pieces of this warp
                for (int base = 0; base < mine; base += kBatch) {
                    float m[kBatch], l[kBatch];
                    float4 x[kBatch];
#pragma unroll
                    for (int u = 0; u < kBatch; ++u) {
                        m[u] = -INFINITY;
                        l[u] = 0.f;
                        x[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                        if (base + u < mine) {
                            const int64_t rr = row0 + static_cast<int64_t>(sub + (base + u) * WPI) * p.n_heads;
                            const float2 ml = __ldcg(reinterpret_cast<const float2 *>(p.ml_part) + rr);
                            m[u] = ml.x;
                            l[u] = ml.y;
                            if (lane < kCols) x[u] = __ldcg(reinterpret_cast<const float4 *>(p.o_part + rr * D) + lane);
                        }
                    }
                    float nM = M;
#pragma unroll
                    for (int u = 0; u < kBatch; ++u) nM = fmaxf(nM, m[u]);
                    const float sc = exp2f(M - nM);   // M = -inf on the first batch: 0
                    acc.x *= sc;
                    acc.y *= sc;
                    acc.z *= sc;
                    acc.w *= sc;
                    L *= sc;
#pragma unroll
                    for (int u = 0; u < kBatch; ++u) {
                        const float w = base + u < mine ? l[u] * exp2f(m[u] - nM) : 0.f;
                        L += w;
                        acc.x = fmaf(w, x[u].x, acc.x);
                        acc.y = fmaf(w, x[u].y, acc.y);
                        acc.z = fmaf(w, x[u].z, acc.z);
                        acc.w = fmaf(w, x[u].w, acc.w);
                    }
                    M = nM;
                }
            }
        }
    }
    if (WPI > 1) {
        if (lane == 0) {
            red_ml[warp][0] = M;
            red_ml[warp][1] = L;
        }
        if (lane < kCols) red_o[warp][lane] = acc;
        __syncthreads();
        if (sub == 0 && merge) {
            float MM = -INFINITY;
#pragma unroll
            for (int u = 0; u < WPI; ++u) MM = fmaxf(MM, red_ml[warp + u][0]);
            float LL = 0.f;
            float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int u = 0; u < WPI; ++u) {
                const float sc = exp2f(red_ml[warp + u][0] - MM);   // a warp without pieces: 0
                LL += red_ml[warp + u][1] * sc;
                if (lane < kCols) {
                    const float4 t = red_o[warp + u][lane];
                    a.x = fmaf(sc, t.x, a.x);
                    a.y = fmaf(sc, t.y, a.y);
                    a.z = fmaf(sc, t.z, a.z);
                    a.w = fmaf(sc, t.w, a.w);
                }
            }
            M = MM;
            L = LL;
            acc = a;
        }
    }
    if (sub == 0 && merge && lane < kCols) {
        const float inv = 1.f / L;
        *reinterpret_cast<__nv_bfloat162 *>(out + lane * 4) = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
        *reinterpret_cast<__nv_bfloat162 *>(out + lane * 4 + 2) = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
    }
}

// Merge of the shared-prefix mode.  One warp per (entry b, head h): the
// pieces are the private role's rows (c + b) for the CTAs c whose range
// meets b's private positions, then the group role's units of member
// u = b % R of group gi = b / R for the CTAs whose range meets the group's
// [gi Ts, gi Ts + Ts).  Both lists follow from T and the shared_roles split,
// as in the split kernel.  An entry shorter than the shared prefix, or with
// metadata that does not fit the partition, is recorded and gets o = 0.
template <int D>
__global__ void __launch_bounds__(256, 4) decode_merge_shared_kernel(const DecodeParams p) {
    constexpr int kCols = D / 4, kBatch = 6;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int item = blockIdx.x * 8 + warp;
    if (item >= p.batch * p.n_heads) return;   // warp-uniform; no block barriers below
    const int b = item / p.n_heads, h = item - b * p.n_heads;
    __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(p.o) + static_cast<int64_t>(item) * D;
    const long long Ts = p.shared_len;
    const int R = p.group_reqs;
    const long long T = __ldg(p.kv_indptr + p.batch);
    const long long lo = __ldg(p.kv_indptr + b), hi = __ldg(p.kv_indptr + b + 1);
    const long long n = hi - lo;
    const int n_cap = min(p.max_len, p.max_ctx_len);
    bool ok = T > 0 && n >= Ts && n == __ldg(p.seq_lens + b) && n <= n_cap && lo >= 0 && hi <= T;
    int np_pr = 0, c_lo = 0, cs_lo = 0, np_sh = 0;
    const int gi = b / R, u = b - (b / R) * R;
    if (ok) {
        const SharedRoles ro = shared_roles(p, T);
        const long long plo = lo - b * Ts, phi = hi - (b + 1) * Ts;   // private range
        if (phi > plo) {
            ok = ro.p_pr_e > 0 && plo >= 0 && phi <= ro.t_pr;
            if (ok) {
                c_lo = part_of(plo, ro.t_pr, ro.p_pr_e);
                np_pr = part_of(phi - 1, ro.t_pr, ro.p_pr_e) - c_lo + 1;
            }
        }
        if (p.group_tc) {   // one partial per chunk of the prefix
            np_sh = p.group_chunks;
        } else {
            cs_lo = part_of(gi * Ts, ro.t_sh, ro.p_sh_e);
            np_sh = part_of((gi + 1) * Ts - 1, ro.t_sh, ro.p_sh_e) - cs_lo + 1;
        }
    }
    // the partials come from the split kernel, which may still run (the
    // piece lists above need only the metadata)
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    if (!ok) {
        if (h == 0 && lane == 0) record_error(p.err, n);
        for (int e = lane; e < D; e += 32) out[e] = __float2bfloat16_rn(0.f);
        return;
    }
    const int np = np_pr + np_sh;
    float M = -INFINITY, L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int base = 0; base < np; base += kBatch) {
        float m[kBatch], l[kBatch];
        float4 x[kBatch];
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
            m[k] = -INFINITY;
            l[k] = 0.f;
            x[k] = make_float4(0.f, 0.f, 0.f, 0.f);
            const int i = base + k;
            if (i < np) {
                const int64_t unit =
                    i < np_pr ? (static_cast<int64_t>(c_lo) + i + b) * p.n_heads + h
                    : p.group_tc
                        ? p.group_unit0 + (static_cast<int64_t>(i - np_pr) * p.batch + b) * p.n_heads + h
                        : p.group_unit0 +
                              ((static_cast<int64_t>(cs_lo) + (i - np_pr) + gi) * R + u) * p.n_heads + h;
                const float2 ml = __ldcg(reinterpret_cast<const float2 *>(p.ml_part) + unit);
                m[k] = ml.x;
                l[k] = ml.y;
                if (lane < kCols) x[k] = __ldcg(reinterpret_cast<const float4 *>(p.o_part + unit * D) + lane);
            }
        }
        float nM = M;
#pragma unroll
        for (int k = 0; k < kBatch; ++k) nM = fmaxf(nM, m[k]);
        const float sc = exp2f(M - nM);
        acc.x *= sc;
        acc.y *= sc;
        acc.z *= sc;
        acc.w *= sc;
        L *= sc;
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
            const float w = base + k < np ? l[k] * exp2f(m[k] - nM) : 0.f;
            L += w;
            acc.x = fmaf(w, x[k].x, acc.x);
            acc.y = fmaf(w, x[k].y, acc.y);
            acc.z = fmaf(w, x[k].z, acc.z);
            acc.w = fmaf(w, x[k].w, acc.w);
        }
        M = nM;
    }
    if (lane < kCols) {
        const float inv = 1.f / L;
        *reinterpret_cast<__nv_bfloat162 *>(out + lane * 4) = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
        *reinterpret_cast<__nv_bfloat162 *>(out + lane * 4 + 2) = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
    }
}

template <int D>
cudaError_t launch_merge_shared(const DecodeParams &p, cudaStream_t s) {
    const int items = p.batch * p.n_heads;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((items + 7) / 8);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_merge_shared_kernel<D>, p);
}

template <int D, int WPI>
cudaError_t launch_merge_wpi(const DecodeParams &p, cudaStream_t s) {
    const int items = p.batch * p.n_heads;
    const int ipc = WPI > 8 ? 1 : 8 / WPI;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((items + ipc - 1) / ipc);
    cfg.blockDim = dim3(WPI > 8 ? 32 * WPI : 256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_merge_balanced_kernel<D, WPI>, p);
}

template <int D>
cudaError_t launch_merge_d(const DecodeParams &p, cudaStream_t s) {
    if (p.shared_len > 0) return launch_merge_shared<D>(p, s);
    // an entry has about (n_parts + batch) / batch pieces: up to 16 warps per
    // entry, each loading its pieces in one or two batches
    const int64_t per_entry = (static_cast<int64_t>(p.n_parts) + p.batch) / (p.batch > 0 ? p.batch : 1);
    int wpi = 1;
    while (wpi < 16 && per_entry > 8 * wpi) wpi *= 2;
    switch (wpi) {
        case 1: return launch_merge_wpi<D, 1>(p, s);
        case 2: return launch_merge_wpi<D, 2>(p, s);
        case 4: return launch_merge_wpi<D, 4>(p, s);
        case 8: return launch_merge_wpi<D, 8>(p, s);
        default: return launch_merge_wpi<D, 16>(p, s);
    }
}

template <int D, int G>
cudaError_t run(const DecodeParams &p, cudaStream_t s) {
    using C = MmaCfg<D>;
    static std::atomic<uint64_t> attr_done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(attr_done.load() & bit)) {
        e = cudaFuncSetAttribute(decode_mma_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(C::kSmem));
        if (e != cudaSuccess) return e;
        attr_done.fetch_or(bit);
    }
    if (p.n_kv_heads == 1 || p.n_kv_heads == 2 || p.n_kv_heads == 4 || p.n_kv_heads == 8)
        return run_hk<D, G>(p, s);
    dim3 grid(p.n_splits, p.n_kv_heads, p.batch);
    decode_mma_kernel<D, G><<<grid, kNT, C::kSmem, s>>>(p);
    return cudaGetLastError();
}

template <int D>
cudaError_t run_group(const DecodeParams &p, int group, cudaStream_t s) {
    switch (group) {
        case 1: return run<D, 1>(p, s);
        case 2: return run<D, 2>(p, s);
        case 4: return run<D, 4>(p, s);
        case 8: return run<D, 8>(p, s);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace

bool decode_balanced_supported(int dtype, int head_dim, int group, int n_kv_heads) {
    return dtype == PKV_BF16 && (head_dim == 64 || head_dim == 128) &&
           (group == 1 || group == 2 || group == 4 || group == 8) &&
           (n_kv_heads == 1 || n_kv_heads == 2 || n_kv_heads == 4 || n_kv_heads == 8);
}

cudaError_t launch_decode_merge_balanced(const DecodeParams &p, int head_dim, cudaStream_t s) {
    return head_dim == 128 ? launch_merge_d<128>(p, s) : launch_merge_d<64>(p, s);
}

cudaError_t launch_decode_split_mma(const DecodeParams &p, int head_dim, int group,
                                    cudaStream_t s) {
    if (p.group_tc) {   // the private role, then the shared prefix on tensor cores as its dependent
        if (head_dim != 128) return cudaErrorNotSupported;
        const cudaError_t e = run_group<128>(p, group, s);
        if (e != cudaSuccess) return e;
        return launch_shared_group_tc(p, group, s);
    }
    return head_dim == 128 ? run_group<128>(p, group, s) : run_group<64>(p, group, s);
}

}  // namespace pkv
