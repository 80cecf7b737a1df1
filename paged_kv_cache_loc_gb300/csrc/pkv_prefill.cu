// pkv_prefill.cu -- ragged paged prefill attention over the token pool.
//
// Operation (AstrAI docs/guides/inference.md, "Attention Backend", prefill
// path): entry b has q_len = qo_indptr[b+1] - qo_indptr[b] new tokens at the
// end of kv_len = kv_indptr[b+1] - kv_indptr[b] positions (prefix P = kv_len -
// q_len, already written).  Packed row qo_indptr[b] + i, head h attends to the
// slots req_to_token[req_pool_indices[b], j] for j <= P + i (causal, the mask
// of astrai/model/transformer.py process_attention_mask) or j < kv_len.
//
// Tiling: one CTA per (query tile, kv head, entry).  A query tile is 64 rows
// of (position, head-in-group) pairs, so the G query heads that share a kv
// head share every gathered K/V tile.  K/V tiles of 64 tokens are gathered
// row-wise through req_to_token with 16-byte cp.async into XOR-swizzled
// shared memory (double buffered), S = Q K^T and O += P V run on bf16 tensor
// cores with fp32 accumulation, with the online softmax in registers.  Tiles
// wholly above the causal diagonal are never loaded; query tiles are issued
// longest-first.
#include <atomic>

#include "pkv_common.cuh"
#include "pkv_launch.h"

namespace pkv {
namespace {

constexpr int kBM = 64;    // rows per CTA (4 warps x 16)
constexpr int kBN = 64;    // kv tokens per tile
constexpr int kNT = 128;

template <int D>
__device__ __forceinline__ int swz(int row, int chunk) {
    return row * D + ((chunk ^ (row & 7)) << 3);
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

template <int D, int G>
struct PrefillCfg {
    static constexpr int kChunks = D / 8;
    static constexpr size_t kSmem = static_cast<size_t>(kBM * D + 4 * kBN * D) * 2;
};

template <int D, int G>
__global__ void __launch_bounds__(kNT) prefill_kernel(const PrefillParams p) {
    using C = PrefillCfg<D, G>;
    using bf16 = __nv_bfloat16;
    extern __shared__ __align__(128) unsigned char smem[];
    bf16 *sQ = reinterpret_cast<bf16 *>(smem);
    bf16 *sK = sQ + kBM * D;          // [2][kBN][D]
    bf16 *sV = sK + 2 * kBN * D;      // [2][kBN][D]

    const int b = blockIdx.z, g = blockIdx.y;
    const int qt = gridDim.x - 1 - blockIdx.x;   // longest causal work first
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    int r = __ldg(p.req_pool_indices + b);
    const int qo0 = __ldg(p.qo_indptr + b);
    const int q_len = __ldg(p.qo_indptr + b + 1) - qo0;
    const int kv_len = __ldg(p.kv_indptr + b + 1) - __ldg(p.kv_indptr + b);
    // q and o hold qo_indptr[batch] packed rows: this entry's rows must lie
    // inside them, or they are neither read nor written
    const long long q_total = __ldg(p.qo_indptr + p.batch);
    const bool rows_ok = qo0 >= 0 && static_cast<long long>(qo0) + q_len <= q_total;
    if (static_cast<unsigned>(r) >= static_cast<unsigned>(p.num_reqs) || q_len < 0 || !rows_ok ||
        q_len > p.max_q_len || kv_len < q_len || kv_len > p.max_ctx_len || kv_len > p.max_kv_len) {
        if (qt == 0 && g == 0 && tid == 0)
            record_error(p.err, static_cast<unsigned>(r) >= static_cast<unsigned>(p.num_reqs) ? r
                                : (q_len >= 0 && !rows_ok) ? qo0 : kv_len);
        return;
    }
    const int rows = q_len * G;
    const int row0 = qt * kBM;
    if (row0 >= rows) return;
    const int P = kv_len - q_len;
    const int pos_last = (min(row0 + kBM, rows) - 1) / G;
    const int kv_end = p.causal ? min(kv_len, P + pos_last + 1) : kv_len;
    const int n_tiles = (kv_end + kBN - 1) / kBN;

    const int64_t slot_stride = static_cast<int64_t>(p.n_kv_heads) * D;
    const bf16 *kbase = static_cast<const bf16 *>(p.k_buffer) + (p.layer_row0 * p.n_kv_heads + g) * D;
    const bf16 *vbase = static_cast<const bf16 *>(p.v_buffer) + (p.layer_row0 * p.n_kv_heads + g) * D;
    const int32_t *r2t = p.req_to_token + static_cast<int64_t>(r) * p.max_ctx_len;

    // Q tile (rows beyond the request are zero-filled)
    {
        const bf16 *qsrc = static_cast<const bf16 *>(p.q);
        for (int idx = tid; idx < kBM * C::kChunks; idx += kNT) {
            const int rr = idx / C::kChunks, c = idx - rr * C::kChunks;
            const int R = row0 + rr;
            bf16 *dst = sQ + swz<D>(rr, c);
            if (R < rows) {
                const int pos = R / G, hh = R - (R / G) * G;
                cp_async16(dst, qsrc + ((static_cast<int64_t>(qo0) + pos) * p.n_heads + g * G + hh) * D + c * 8);
            } else {
                cp_async16(dst, qsrc, 0);
            }
        }
    }
    auto load_kv = [&](int tile, int buf) {
        const int kv0 = tile * kBN;
        bf16 *dk = sK + buf * kBN * D;
        bf16 *dv = sV + buf * kBN * D;
#pragma unroll 4
        for (int idx = tid; idx < 2 * kBN * C::kChunks; idx += kNT) {
            const int is_v = idx / (kBN * C::kChunks);
            const int rem = idx - is_v * (kBN * C::kChunks);
            const int t = rem / C::kChunks, c = rem - t * C::kChunks;
            const int j = kv0 + t;
            bf16 *dst = (is_v ? dv : dk) + swz<D>(t, c);
            if (j < kv_end) {
                int slot = __ldg(r2t + j);
                if (static_cast<unsigned long long>(static_cast<long long>(slot)) >=
                    static_cast<unsigned long long>(p.size)) {
                    record_error(p.err, slot);
                    slot = 0;
                }
                cp_async16(dst, (is_v ? vbase : kbase) + slot * slot_stride + c * 8);
            } else {
                cp_async16(dst, kbase, 0);
            }
        }
    };
    load_kv(0, 0);
    cp_async_commit();

    // this thread's two fragment rows
    const int rA = warp * 16 + (lane >> 2), rB = rA + 8;
    const int RA = row0 + rA, RB = row0 + rB;
    const int limA = RA < rows ? (p.causal ? P + RA / G : kv_len - 1) : -1;
    const int limB = RB < rows ? (p.causal ? P + RB / G : kv_len - 1) : -1;

    float o_acc[D / 8][4];
#pragma unroll
    for (int i = 0; i < D / 8; ++i) o_acc[i][0] = o_acc[i][1] = o_acc[i][2] = o_acc[i][3] = 0.f;
    float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;
    uint32_t qa[D / 16][4];

    for (int tile = 0; tile < n_tiles; ++tile) {
        cp_async_wait<0>();
        __syncthreads();
        if (tile == 0) {
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
                ldsm_x4(qa[ks], sQ + swz<D>(warp * 16 + (lane & 15), 2 * ks + (lane >> 4)));
        }
        if (tile + 1 < n_tiles) load_kv(tile + 1, (tile + 1) & 1);
        cp_async_commit();

        const bf16 *k = sK + (tile & 1) * kBN * D;
        const bf16 *v = sV + (tile & 1) * kBN * D;
        float s[kBN / 8][4];
#pragma unroll
        for (int i = 0; i < kBN / 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
            for (int np = 0; np < kBN / 16; ++np) {
                uint32_t kb[4];
                ldsm_x4(kb, k + swz<D>(np * 16 + ((lane >> 4) & 1) * 8 + (lane & 7),
                                       2 * ks + ((lane >> 3) & 1)));
                mma16816(s[2 * np], qa[ks], kb[0], kb[1]);
                mma16816(s[2 * np + 1], qa[ks], kb[2], kb[3]);
            }
        }

        // scale, mask, online softmax (base 2)
        const int kv0 = tile * kBN;
        float mxA = -INFINITY, mxB = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < kBN / 8; ++nt) {
            const int j = kv0 + nt * 8 + (lane & 3) * 2;
            s[nt][0] = j <= limA ? s[nt][0] * p.scale_log2 : -INFINITY;
            s[nt][1] = j + 1 <= limA ? s[nt][1] * p.scale_log2 : -INFINITY;
            s[nt][2] = j <= limB ? s[nt][2] * p.scale_log2 : -INFINITY;
            s[nt][3] = j + 1 <= limB ? s[nt][3] * p.scale_log2 : -INFINITY;
            mxA = fmaxf(mxA, fmaxf(s[nt][0], s[nt][1]));
            mxB = fmaxf(mxB, fmaxf(s[nt][2], s[nt][3]));
        }
        mxA = fmaxf(mxA, __shfl_xor_sync(0xffffffffu, mxA, 1));
        mxA = fmaxf(mxA, __shfl_xor_sync(0xffffffffu, mxA, 2));
        mxB = fmaxf(mxB, __shfl_xor_sync(0xffffffffu, mxB, 1));
        mxB = fmaxf(mxB, __shfl_xor_sync(0xffffffffu, mxB, 2));
        const float mnA = fmaxf(mA, mxA), mnB = fmaxf(mB, mxB);
        const float uA = mnA == -INFINITY ? 0.f : mnA;   // fully masked so far
        const float uB = mnB == -INFINITY ? 0.f : mnB;
        const float alA = exp2f(mA - uA), alB = exp2f(mB - uB);
        mA = mnA;
        mB = mnB;
        float sumA = 0.f, sumB = 0.f;
#pragma unroll
        for (int nt = 0; nt < kBN / 8; ++nt) {
            s[nt][0] = exp2f(s[nt][0] - uA);
            s[nt][1] = exp2f(s[nt][1] - uA);
            s[nt][2] = exp2f(s[nt][2] - uB);
            s[nt][3] = exp2f(s[nt][3] - uB);
            sumA += s[nt][0] + s[nt][1];
            sumB += s[nt][2] + s[nt][3];
        }
        lA = lA * alA + sumA;
        lB = lB * alB + sumB;
#pragma unroll
        for (int i = 0; i < D / 8; ++i) {
            o_acc[i][0] *= alA;
            o_acc[i][1] *= alA;
            o_acc[i][2] *= alB;
            o_acc[i][3] *= alB;
        }

        // O += P V
#pragma unroll
        for (int kt = 0; kt < kBN / 16; ++kt) {
            uint32_t pa[4];
            pa[0] = pack_bf16(s[2 * kt][0], s[2 * kt][1]);
            pa[1] = pack_bf16(s[2 * kt][2], s[2 * kt][3]);
            pa[2] = pack_bf16(s[2 * kt + 1][0], s[2 * kt + 1][1]);
            pa[3] = pack_bf16(s[2 * kt + 1][2], s[2 * kt + 1][3]);
#pragma unroll
            for (int dp = 0; dp < D / 16; ++dp) {
                uint32_t vb[4];
                ldsm_x4_t(vb, v + swz<D>(kt * 16 + ((lane >> 3) & 1) * 8 + (lane & 7),
                                         2 * dp + ((lane >> 4) & 1)));
                mma16816(o_acc[2 * dp], pa, vb[0], vb[1]);
                mma16816(o_acc[2 * dp + 1], pa, vb[2], vb[3]);
            }
        }
    }
    cp_async_wait<0>();

    lA += __shfl_xor_sync(0xffffffffu, lA, 1);
    lA += __shfl_xor_sync(0xffffffffu, lA, 2);
    lB += __shfl_xor_sync(0xffffffffu, lB, 1);
    lB += __shfl_xor_sync(0xffffffffu, lB, 2);
    bf16 *out = static_cast<bf16 *>(p.o);
    if (RA < rows) {
        const int pos = RA / G, hh = RA - (RA / G) * G;
        bf16 *orow = out + ((static_cast<int64_t>(qo0) + pos) * p.n_heads + g * G + hh) * D;
        const float inv = 1.f / lA;
#pragma unroll
        for (int i = 0; i < D / 8; ++i)
            *reinterpret_cast<uint32_t *>(orow + i * 8 + (lane & 3) * 2) =
                pack_bf16(o_acc[i][0] * inv, o_acc[i][1] * inv);
    }
    if (RB < rows) {
        const int pos = RB / G, hh = RB - (RB / G) * G;
        bf16 *orow = out + ((static_cast<int64_t>(qo0) + pos) * p.n_heads + g * G + hh) * D;
        const float inv = 1.f / lB;
#pragma unroll
        for (int i = 0; i < D / 8; ++i)
            *reinterpret_cast<uint32_t *>(orow + i * 8 + (lane & 3) * 2) =
                pack_bf16(o_acc[i][2] * inv, o_acc[i][3] * inv);
    }
}

template <int D, int G>
cudaError_t run(const PrefillParams &p, cudaStream_t s) {
    using C = PrefillCfg<D, G>;
    static std::atomic<uint64_t> attr_done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(attr_done.load() & bit)) {
        e = cudaFuncSetAttribute(prefill_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(C::kSmem));
        if (e != cudaSuccess) return e;
        attr_done.fetch_or(bit);
    }
    const int qtiles = (p.max_q_len * G + kBM - 1) / kBM;
    dim3 grid(qtiles, p.n_kv_heads, p.batch);
    prefill_kernel<D, G><<<grid, kNT, C::kSmem, s>>>(p);
    return cudaGetLastError();
}

template <int D>
cudaError_t run_group(const PrefillParams &p, int group, cudaStream_t s) {
    switch (group) {
        case 1: return run<D, 1>(p, s);
        case 2: return run<D, 2>(p, s);
        case 4: return run<D, 4>(p, s);
        case 8: return run<D, 8>(p, s);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace

bool prefill_supported(int dtype, int head_dim, int group) {
    return dtype == PKV_BF16 && (head_dim == 64 || head_dim == 128) &&
           (group == 1 || group == 2 || group == 4 || group == 8);
}

cudaError_t launch_prefill(const PrefillParams &p, int dtype, int head_dim, int group,
                           cudaStream_t s) {
    if (!prefill_supported(dtype, head_dim, group)) return cudaErrorNotSupported;
    if (p.batch == 0 || p.max_q_len == 0) return cudaSuccess;
    if (prefill_tc_supported(dtype, head_dim, group)) return launch_prefill_tc(p, group, s);
    return head_dim == 128 ? run_group<128>(p, group, s) : run_group<64>(p, group, s);
}

}  // namespace pkv
