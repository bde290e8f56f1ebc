// Tensor-core paged attention in the transposed form, for head_dim 256 (bf16 / f16), sm_103a.
//
// The 16-row tiles of attn_mma.cu would hold, at head_dim 256, 64 registers of query fragments and
// 128 of output accumulators per thread.  This kernel computes S^T = K Q^T and O^T = V^T P^T
// instead: keys and the head dimension sit on the MMA's 16-row side and 8 query rows on its 8-wide
// side, so a thread holds 32 registers of Q^T and 64 of O^T.  Units are (sequence, kv head, split,
// 8 query rows); a longer query run takes several units, each reading the keys again.
//
// Staging, split plan, masking and the softmax guards are those of the decode kernel: the
// producer warp walks the unit's pages (one 4-D TMA box per page and pool into a ring of 64-key
// stages, 128-byte swizzled), and consumer warp w takes keys [16 w, 16 w + 16) of every stage:
//   * A = K rows by ldmatrix, B = Q^T from registers: S^T for 16 keys x 8 rows;
//   * online softmax per query row (rocMLIR PR #2371 guards: a running max of -inf is replaced by 0
//     before exp2, and a row whose sum is 0 stores 0 / lse -inf), P split into a 16-bit high part
//     and its rounding remainder, P^T turned into the B operand with movmatrix;
//   * A = V^T by the transposing ldmatrix: O^T += V^T (Ph + Pl)^T.
// The four warps' softmax states are merged through shared memory at the end.
#include "mma_common.cuh"

namespace pa {

using namespace mmac;

namespace {

constexpr int kTRows = 8;  // query rows of one unit

__device__ __forceinline__ uint32_t movmatrix_trans16(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

}  // namespace

template <typename T, int D, int NSTAGE>
__global__ void __launch_bounds__(kMmaThreads, 1)
    paged_attn_mma_t_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                            const FwdParams p, int ps_shift) {
    using Op = MmaOp<T>;
    constexpr int kStage = Geo<D>::kStageBytes;
    constexpr int kChunks = Geo<D>::kChunks;
    constexpr int MT = D / 16;  // 16-wide head-dim tiles

    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bars[3 * NSTAGE];

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int ps = 1 << ps_shift;
    int unit = blockIdx.x;
    const int rt = unit % p.row_tiles;
    unit /= p.row_tiles;
    const int kvh = unit % p.Hkv;
    unit /= p.Hkv;
    const int s = unit % p.split_kv;
    const int b = unit / p.split_kv;
    const SeqRows sq = uniform_seq(p, b);

    int L = max(p.seq_lens[b], 0);
    if (L > p.W * ps) {  // never read past the sequence's block-table row
        if (threadIdx.x == 0) atomicOr(p.err, (unsigned int)PA_ERRBIT_SEQ_CLIPPED);
        L = p.W * ps;
    }
    int pg0, pg1;
    split_pages(L, ps, p.split_kv, s, pg0, pg1);
    const int k_lo = pg0 * ps;
    const int k_hi_split = min(pg1 * ps, L);
    const int row0 = rt * kTRows;
    const int row_end = min(row0 + kTRows, p.rows);
    const int k_hi = min(k_hi_split, row_key_limit(p, b, L, (row_end - 1) / p.G));
    const int n_tiles = k_hi > k_lo ? (k_hi - k_lo + kMmaTileKeys - 1) / kMmaTileKeys : 0;
    if (n_tiles == 0) {
        if (warp < kMmaConsumerWarps) store_empty_unit<T, D>(p, sq, kvh, s, row0, row_end);
        return;
    }

    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    const uint32_t bar_fk = smem_u32(&bars[0]);
    const uint32_t bar_fv = smem_u32(&bars[NSTAGE]);
    const uint32_t bar_em = smem_u32(&bars[2 * NSTAGE]);
    if (threadIdx.x == 0) {
        for (int st = 0; st < NSTAGE; ++st) {
            mbar_init(bar_fk + 8 * st, 1);
            mbar_init(bar_fv + 8 * st, 1);
            mbar_init(bar_em + 8 * st, kMmaConsumerWarps);
        }
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == kMmaConsumerWarps) {
        produce_pages16<D, NSTAGE>(&tmK, &tmV, p, b, kvh, pg0, k_hi, n_tiles, ps_shift, sbase, bar_fk, bar_fv, bar_em,
                                   lane);
        return;
    }

    // ==================================================================== consumers
    const int g = lane >> 2;
    const int tq = lane & 3;
    const int kw0 = warp * 16;  // this warp's keys in every stage
    // Q^T operands: this lane's row row0 + g, head-dim pairs 16 kk + 2 tq (b0) and + 8 (b1).  The
    // score and output fragments hold rows row0 + 2 tq + e (e = 0, 1).
    uint32_t qb[MT][2];
    {
        const int r = row0 + g;
        const bool valid = r < row_end;
        const T *q = reinterpret_cast<const T *>(p.q) + (valid ? q_row_offset(p, out_row_index(p, sq, kvh, r)) : 0);
#pragma unroll
        for (int kk = 0; kk < MT; ++kk) {
            qb[kk][0] = valid ? __ldg(reinterpret_cast<const uint32_t *>(q + 16 * kk + 2 * tq)) : 0u;
            qb[kk][1] = valid ? __ldg(reinterpret_cast<const uint32_t *>(q + 16 * kk + 8 + 2 * tq)) : 0u;
        }
    }
    int lim[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int rc = row0 + 2 * tq + e;
        lim[e] = rc < row_end ? min(k_hi_split, row_key_limit(p, b, L, rc / p.G)) : k_lo;
    }
    // keys at or past the furthest limit of the unit's rows are masked for all of them
    const int key_lim = min(k_hi, (int)__reduce_max_sync(0xffffffffu, (unsigned)max(lim[0], lim[1])));

    float m[2] = {kNegInf, kNegInf}, l[2] = {0.f, 0.f};
    float acc[MT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
    // ldmatrix row addresses: K (keys along M) and V (keys along k after the transpose)
    const int key_k = kw0 + (lane & 7) + (((lane >> 3) & 1) << 3);
    const int ck = lane >> 4;
    const int key_v = kw0 + (lane & 7) + (((lane >> 4) & 1) << 3);
    const int cv = (lane >> 3) & 1;

    bool bad = false;
    for (int t = 0; t < n_tiles; ++t) {
        const int st = t % NSTAGE;
        const uint32_t par = (t / NSTAGE) & 1;
        const uint32_t kbuf = sbase + (uint32_t)(st * 2 * kStage);
        const uint32_t vbuf = kbuf + kStage;
        const int tile_k0 = k_lo + t * kMmaTileKeys;
        const bool active = tile_k0 + kw0 < key_lim;  // warp-uniform

        if (!bad) {
            const bool ok = mbar_wait(bar_fk + 8 * st, par, p.err);
            bad = __any_sync(0xffffffffu, !ok);
        }
        uint32_t pb[2][2];  // P^T operands: [high / low part][keys 0-7 / 8-15]
        float al[2] = {1.f, 1.f};
        if (!bad && active) {
            // ---- S^T = K Q^T: two partial sums over alternating head-dim steps
            float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
            for (int kk = 0; kk < MT; ++kk) {
                uint32_t a[4];
                ldmatrix_x4(kv_chunk_addr<D>(kbuf, key_k, 2 * kk + ck, ps_shift), a[0], a[1], a[2], a[3]);
                Op::run(sc[kk & 1], a, qb[kk][0], qb[kk][1]);
            }
            // ---- mask, scale (log2 domain), online softmax per row: keys g / g + 8, rows 2 tq + e
            const int j0 = tile_k0 + kw0 + g;
            float pv[2][2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                float x0 = sc[0][e] + sc[1][e];
                float x1 = sc[0][2 + e] + sc[1][2 + e];
                x0 = (j0 < lim[e]) ? x0 * p.scale_log2 : kNegInf;
                x1 = (j0 + 8 < lim[e]) ? x1 * p.scale_log2 : kNegInf;
                float mx = fmaxf(x0, x1);
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                const float mn = fmaxf(m[e], mx);
                // -inf - (-inf) guard: an all-masked row keeps max -inf and uses 0 as its offset
                const float mu = (mn == kNegInf) ? 0.f : mn;
                al[e] = exp2f(m[e] - mu);
                m[e] = mn;
                pv[e][0] = exp2f(x0 - mu);
                pv[e][1] = exp2f(x1 - mu);
                l[e] = l[e] * al[e] + (pv[e][0] + pv[e][1]);
            }
            // P^T tiles (rows: keys g / g + 8; columns: rows 2 tq, 2 tq + 1), high part and remainder,
            // transposed into the B operand layout (keys along k)
            const uint32_t h0 = Op::pack(pv[0][0], pv[1][0]);
            const uint32_t h1 = Op::pack(pv[0][1], pv[1][1]);
            const float2 u0 = Op::unpack(h0), u1 = Op::unpack(h1);
            const uint32_t r0 = Op::pack(pv[0][0] - u0.x, pv[1][0] - u0.y);
            const uint32_t r1 = Op::pack(pv[0][1] - u1.x, pv[1][1] - u1.y);
            pb[0][0] = movmatrix_trans16(h0);
            pb[0][1] = movmatrix_trans16(h1);
            pb[1][0] = movmatrix_trans16(r0);
            pb[1][1] = movmatrix_trans16(r1);
            if (__any_sync(0xffffffffu, al[0] != 1.f || al[1] != 1.f)) {  // a running max moved
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    acc[mt][0] *= al[0];
                    acc[mt][1] *= al[1];
                    acc[mt][2] *= al[0];
                    acc[mt][3] *= al[1];
                }
            }
        }
        if (!bad) {
            const bool ok = mbar_wait(bar_fv + 8 * st, par, p.err);
            bad = __any_sync(0xffffffffu, !ok);
        }
        if (!bad && active && tile_k0 + kMmaTileKeys > k_hi) {
            // Last stage: V rows at or past k_hi (past the sequence, or pages never loaded) may hold
            // any bits; their weight is 0, but 0 x NaN is NaN, so zero this warp's such rows.
            for (int idx = lane; idx < 16 * kChunks; idx += 32) {
                const int key = kw0 + idx / kChunks;
                if (tile_k0 + key >= k_hi) {
                    const uint32_t a = kv_chunk_addr<D>(vbuf, key, idx % kChunks, ps_shift);
                    asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0u) : "memory");
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
        }
        if (!bad && active) {
            // ---- O^T += V^T (Ph + Pl)^T over the warp's 16 keys
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                uint32_t a[4];
                ldmatrix_x4_trans(kv_chunk_addr<D>(vbuf, key_v, 2 * mt + cv, ps_shift), a[0], a[1], a[2], a[3]);
                Op::run(acc[mt], a, pb[0][0], pb[0][1]);
                Op::run(acc[mt], a, pb[1][0], pb[1][1]);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_em + 8 * st);
    }

    // row sums over the 8 key lanes of each row
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        l[e] += __shfl_xor_sync(0xffffffffu, l[e], 4);
        l[e] += __shfl_xor_sync(0xffffffffu, l[e], 8);
        l[e] += __shfl_xor_sync(0xffffffffu, l[e], 16);
    }
    // ---- merge the four warps' states through shared memory (reuses the ring)
    constexpr int ACC_STRIDE = D + 4;
    float *sm = reinterpret_cast<float *>(smem_raw + (sbase - raw));
    named_bar_sync(1, kMmaConsumerWarps * 32);  // every warp is done reading the ring
    {
        float *wa = sm + warp * 16 * ACC_STRIDE;
        float *s_m = sm + kMmaConsumerWarps * 16 * ACC_STRIDE;
        float *s_l = s_m + kMmaConsumerWarps * 16;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int r = 2 * tq + e;
                wa[r * ACC_STRIDE + 16 * mt + g] = acc[mt][e];
                wa[r * ACC_STRIDE + 16 * mt + g + 8] = acc[mt][2 + e];
            }
        if (g == 0) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                s_m[warp * 16 + 2 * tq + e] = m[e];
                s_l[warp * 16 + 2 * tq + e] = l[e];
            }
        }
    }
    named_bar_sync(1, kMmaConsumerWarps * 32);
    if (!bad) decode_merge_store<T, D>(p, sm, sq, kvh, s, row0, row_end);
}

// ------------------------------------------------------------------------ host side
template <typename T, int D, int NSTAGE>
static cudaError_t launch_mma_t_t(const FwdParams &p, const CUtensorMap &tmk, const CUtensorMap &tmv,
                                  cudaStream_t stream) {
    constexpr size_t smem = (size_t)NSTAGE * 2 * Geo<D>::kStageBytes + 1024;
    static_assert(merge_scratch_bytes(D) + 1024 <= smem, "merge scratch must fit in the ring");
    auto kern = paged_attn_mma_t_kernel<T, D, NSTAGE>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int ps_shift = 0;
    while ((1 << ps_shift) < p.ps) ++ps_shift;
    FwdParams q = p;
    q.row_tiles = (p.rows + kTRows - 1) / kTRows;
    const long long units = (long long)p.B * p.split_kv * p.Hkv * q.row_tiles;
    if (units <= 0) return cudaSuccess;
    if (units > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    kern<<<(unsigned)units, kMmaThreads, smem, stream>>>(tmk, tmv, q, ps_shift);
    return cudaGetLastError();
}

cudaError_t launch_mma_t(const FwdParams &p, int dtype, const CUtensorMap &tmk, const CUtensorMap &tmv,
                         cudaStream_t stream) {
    if (p.D != 256) return cudaErrorInvalidValue;
    if (dtype == PA_BF16) return launch_mma_t_t<__nv_bfloat16, 256, 3>(p, tmk, tmv, stream);
    return launch_mma_t_t<__half, 256, 3>(p, tmk, tmv, stream);
}

}  // namespace pa
