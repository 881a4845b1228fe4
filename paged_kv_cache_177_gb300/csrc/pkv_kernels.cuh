// pkv_kernels.cuh -- device code of the PagedAttention decode library.
//
// K1 decode_bf16_kernel   block-table gather (TMA) + QK^T + online softmax + PV on tensor cores
// K1 decode_f32_staged_kernel  the same step for fp32 caches on the CUDA cores (exact-precision path)
// K2 lse_reduce_kernel    merges split-context partitions with a log-sum-exp reduce
// K3 kv_append_kernel     slot-mapped write of new tokens' K/V
// K4 move_blocks_kernel   whole-block copies: copy-on-write, swap to/from a host pool, several layers
// K5 validate_*_kernel    device-side range checks of the metadata
//
// The method ("PagedAttention: gestionar la KV cache como memoria de un
// sistema operativo", josueisai.com, section "Cómo funciona por dentro"):
// attention walks a sequence's block table in logical order, reading each
// physical block's keys and values, and returns the softmax-weighted sum of
// the values. Blocks hold 16 tokens ("Batching Continuo y PagedAttention",
// cruxr.ai, section "PagedAttention: Memoria virtual para la KV cache").
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <climits>

#include "pagedkv.h"
#include "pkv_ptx.cuh"

namespace pkv {

constexpr int kBlock = 16;  // tokens per physical block
// Softmax weights are rounded to bf16 for the P V product. When only a few
// comparable weights make up a row and their V rows cancel, that rounding
// alone moves the output by up to ~3e-3 absolute; once a row spans 64 tokens
// or more the per-weight errors average out. So the weights of the first
// kSplitBlocks blocks of every sequence (positions 0..63) enter the product
// as hi + lo, two bf16 values (16 significant bits), at the cost of a second
// P V product for those blocks only.
constexpr int kSplitBlocks = 4;

// Device error word (PKV_DEVERR_* bits), read back by pkv_device_error().
__device__ unsigned int g_dev_error = 0;

__device__ __forceinline__ void raise_error(unsigned int bits) { atomicOr(&g_dev_error, bits); }

// Output element from the fp32 result: bf16 rounded to nearest even, or the
// fp32 value itself (bf16 inputs with fp32 output: the accumulator before
// rounding, for error analysis).
template <typename OutT>
__device__ __forceinline__ OutT to_out(float v) {
    if constexpr (sizeof(OutT) == 2) return __float2bfloat16_rn(v);
    else return v;
}

struct DecodeParams {
    void *out;                    // [S][Hq][D]
    const void *q;                // [S][Hq][D]
    const void *k_cache;          // [NB][Hkv][16][D] (fp32 path; bf16 path reads through tensor maps)
    const void *v_cache;
    const int32_t *block_tables;  // [S][maxB]
    const int32_t *context_lens;  // [S]
    float *ws_ml;                 // [S][Hq][max_parts][2]: running max (log2 domain), sum
    float *ws_o;                  // [S][Hq][max_parts][D]: partition output, normalised by its own sum
    float scale_log2;             // scale * log2(e): scores are kept in the log2 domain
    int num_seqs, num_q_heads, num_kv_heads, group;
    int max_blocks_per_seq, num_blocks, max_context_len;
    int part_blocks;              // blocks per split-context partition
    int max_parts;                // partitions allotted per (sequence, head) in the workspace
    int *counters;                // persistent kernel: one arrival counter per worker (indexed by the
                                  // first worker of a cut unit), zero between calls;
                                  // shared-prefix kernel: [groups] partitions of each group's union
    float *partials;              // persistent kernel: [workers][2][g][2 + D] segment states
    // shared-prefix (cascade) decode
    const int32_t *group_members; // [num_groups][group_size] sequence ids, -1 = empty
    const int32_t *shared_blocks; // [num_groups] leading blocks the members share
    int num_groups, group_size;
    int pre_parts;                // workspace slots per row reserved for the prefix parts
};


// A sequence's usable length: negative lengths and lengths past the table or
// past max_context_len are clamped (and flagged by thread 0 of one CTA).
__device__ __forceinline__ int seq_len(const DecodeParams &p, int s, bool flag) {
    int len = __ldg(p.context_lens + s);
    const int cap = min(p.max_blocks_per_seq * kBlock, p.max_context_len);
    if (len < 0 || len > cap) {
        if (flag) raise_error(PKV_DEVERR_LENGTH);
        len = len < 0 ? 0 : cap;
    }
    return len;
}

// Sum or max over the CTA (all threads call it; scratch holds 32 floats).
__device__ __forceinline__ float block_reduce(float v, bool is_max, float *scratch) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float w = __shfl_xor_sync(0xffffffffu, v, o);
        v = is_max ? fmaxf(v, w) : v + w;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    __syncthreads();
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    v = is_max ? -INFINITY : 0.f;
    for (int w = 0; w < nw; ++w) v = is_max ? fmaxf(v, scratch[w]) : v + scratch[w];
    return v;
}



// =====================================================================================
// The per-block step shared by both bf16 decode kernels. One warp attends a
// (block, kv head) tile already staged in shared memory (K and V, [16][D]
// each, 128-byte swizzle) for the g query heads of the group:
//   S^T[16 tok x 8 heads]  = K[16 x D] . Q^T[D x 8]       (mma m16n8k16, bf16)
//   m' = max(m, max_t s_t);  p_t = 2^(s_t - m');  l = l 2^(m - m') + sum_t p_t
//   O^T[D x 8 heads]      = O^T 2^(m - m') + V^T[D x 16] . P^T[16 x 8]
// The query heads of a GQA group share the tile, which is read from HBM once
// per group; the group (padded to 8 or 16) is the MMA's N. Scores are kept in
// the log2 domain (scale_log2 = scale log2 e). Lane (gq = lane/4, t4 = lane%4)
// holds heads 2 t4, 2 t4 + 1 of each 8-wide n-tile.
// =====================================================================================
template <int D, int NT>
struct WarpAttn {
    static constexpr int kSteps = D / 16;
    static constexpr int kSubBytes = kBlock * 128;      // 2 KiB: 16 rows of 64 bf16
    static constexpr int kSub = D / 64;
    using QFrag = uint32_t[kSteps][NT][2];
    using Scores = float[NT][4];
    float m[NT][2], l[NT][2];
    float acc[kSteps][NT][4];
    QFrag qf;                                            // Q^T as the MMA B operand

    __device__ __forceinline__ void set_q(const QFrag &f) {
#pragma unroll
        for (int kk = 0; kk < kSteps; ++kk)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                qf[kk][nt][0] = f[kk][nt][0];
                qf[kk][nt][1] = f[kk][nt][1];
            }
    }

    // Writes the g heads' outputs O / l (after reduce_l); out_rows = [g][D].
    template <typename OutT>
    __device__ __forceinline__ void store_rows(OutT *out_rows, int g, int lane) const {
        const int gq = lane >> 2, t4 = lane & 3;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int head = nt * 8 + 2 * t4 + (e & 1);
                if (head < g) {
                    const float inv = 1.f / l[nt][e & 1];
#pragma unroll
                    for (int mt = 0; mt < kSteps; ++mt)
                        out_rows[(size_t)head * D + 16 * mt + gq + (e >> 1) * 8] = to_out<OutT>(acc[mt][nt][e] * inv);
                }
            }
    }

    // Writes every column's (max, sum) into ml [8 NT][2] and unnormalised
    // acc into the rows of acc_rows [8 NT][stride] (after reduce_l), for a
    // merge of several warps' states.
    __device__ __forceinline__ void store_merge(float *ml, float *acc_rows, int stride, int lane) const {
        const int gq = lane >> 2, t4 = lane & 3;
        if (gq == 0) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const int head = nt * 8 + 2 * t4 + c;
                    ml[head * 2 + 0] = m[nt][c];
                    ml[head * 2 + 1] = l[nt][c];
                }
        }
#pragma unroll
        for (int mt = 0; mt < kSteps; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int head = nt * 8 + 2 * t4 + (e & 1);
                    acc_rows[head * stride + 16 * mt + gq + (e >> 1) * 8] = acc[mt][nt][e];
                }
    }

    // Writes the g heads' (max, sum, unnormalised acc) states (after
    // reduce_l); slot = [g][2 + D].
    __device__ __forceinline__ void store_state(float *slot, int g, int lane) const {
        const int gq = lane >> 2, t4 = lane & 3;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int head = nt * 8 + 2 * t4 + (e & 1);
                if (head < g) {
                    float *row = slot + (size_t)head * (2 + D);
                    if (gq == 0 && e < 2) {
                        row[0] = m[nt][e];
                        row[1] = l[nt][e];
                    }
#pragma unroll
                    for (int mt = 0; mt < kSteps; ++mt) row[2 + 16 * mt + gq + (e >> 1) * 8] = acc[mt][nt][e];
                }
            }
    }

    __device__ __forceinline__ void reset() {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            m[nt][0] = m[nt][1] = -INFINITY;
            l[nt][0] = l[nt][1] = 0.f;
#pragma unroll
            for (int mt = 0; mt < kSteps; ++mt)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[mt][nt][e] = 0.f;
        }
    }

    // b0 = q[head gq][16kk + 2t4 .. +1], b1 = the same + 8; heads past g read as 0.
    static __device__ __forceinline__ void load_q_frags(uint32_t (&f)[kSteps][NT][2], const __nv_bfloat16 *q_group,
                                                        int g, int lane) {
        const int gq = lane >> 2, t4 = lane & 3;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int hl = nt * 8 + gq;
            const bool hv = hl < g;
            const uint32_t *qrow = reinterpret_cast<const uint32_t *>(q_group + (size_t)(hv ? hl : 0) * D);
#pragma unroll
            for (int kk = 0; kk < kSteps; ++kk) {
                f[kk][nt][0] = hv ? __ldg(qrow + (16 * kk + 2 * t4) / 2) : 0u;
                f[kk][nt][1] = hv ? __ldg(qrow + (16 * kk + 8 + 2 * t4) / 2) : 0u;
            }
        }
    }

    __device__ __forceinline__ void load_q(const __nv_bfloat16 *q_group, int g, int lane) {
        load_q_frags(qf, q_group, g, lane);
    }

    // Columns gathered from any query rows: row_of(column) is the row index
    // into q ([rows][D]) of MMA column `column`, or -1 for an unused column.
    template <class RowOf>
    __device__ __forceinline__ void load_q_rows(const __nv_bfloat16 *q, RowOf row_of, int lane) {
        const int gq = lane >> 2, t4 = lane & 3;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int row = row_of(nt * 8 + gq);
            const uint32_t *qrow = reinterpret_cast<const uint32_t *>(q + (size_t)(row >= 0 ? row : 0) * D);
#pragma unroll
            for (int kk = 0; kk < kSteps; ++kk) {
                qf[kk][nt][0] = row >= 0 ? __ldg(qrow + (16 * kk + 2 * t4) / 2) : 0u;
                qf[kk][nt][1] = row >= 0 ? __ldg(qrow + (16 * kk + 8 + 2 * t4) / 2) : 0u;
            }
        }
    }

    // Attends one staged tile: sk, sv = shared addresses of the K and V tiles.
    // Rows below `lo` are not tokens of the sequence: the last block of a
    // sequence with v valid tokens is loaded shifted down by lo = 16 - v rows,
    // so its first lo rows arrive zero-filled (zero V rows cannot poison the
    // product) and are masked out of the softmax here.
    // col_lo, col_hi: the MMA columns this block is attended for (columns
    // outside get no weight from it; a shared-prefix unit attends each
    // member's own blocks for that member's columns only).
    __device__ __forceinline__ void block(uint32_t sk, uint32_t sv, int lo, float scale_log2, int lane,
                                          int col_lo = 0, int col_hi = 8 * NT, bool split = false) {
        float sc[NT][4];
        scores(sk, sc, lane);
        softmax_pv(sc, sv, lo, scale_log2, lane, col_lo, col_hi, split);
    }

    // S^T = K . Q^T for the 16 tokens of the staged K tile (two independent
    // accumulation chains over the head dimension, summed at the end).
    __device__ __forceinline__ void scores(uint32_t sk, float (&sc)[NT][4], int lane) const {
        const int mi = lane >> 3, r8 = lane & 7;
        float sb[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) sc[nt][e] = sb[nt][e] = 0.f;
#pragma unroll
        for (int kk = 0; kk < kSteps; ++kk) {
            const int u = kk >> 2;
            const int row = r8 + (mi & 1) * 8;
            const int chunk = (kk & 3) * 2 + (mi >> 1);
            uint32_t a[4];
            ldsm_x4(sk + u * kSubBytes + row * 128 + ((chunk ^ (row & 7)) << 4), a);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                if (kk & 1)
                    mma_bf16_16816(sb[nt], a, qf[kk][nt][0], qf[kk][nt][1]);
                else
                    mma_bf16_16816(sc[nt], a, qf[kk][nt][0], qf[kk][nt][1]);
            }
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) sc[nt][e] += sb[nt][e];
    }

    // Online-softmax update with the block's scores, then O^T += V^T . P^T
    // from the staged V tile. With `split` the weights enter the product as
    // the sum of two bf16 values (the rounded weight and its rounding
    // remainder), 16 significant bits instead of 8 (see kSplitBlocks).
    __device__ __forceinline__ void softmax_pv(const float (&sc)[NT][4], uint32_t sv, int lo, float scale_log2,
                                               int lane, int col_lo = 0, int col_hi = 8 * NT, bool split = false) {
        const int gq = lane >> 2, t4 = lane & 3;
        const int mi = lane >> 3, r8 = lane & 7;
        const bool v0 = gq >= lo, v1 = gq + 8 >= lo;
        uint32_t pb0[NT], pb1[NT], pl0[NT], pl1[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int c0 = nt * 8 + 2 * t4;
            const bool k0 = c0 >= col_lo && c0 < col_hi, k1 = c0 + 1 >= col_lo && c0 + 1 < col_hi;
            const float x0 = (v0 && k0) ? sc[nt][0] * scale_log2 : -INFINITY;
            const float x1 = (v0 && k1) ? sc[nt][1] * scale_log2 : -INFINITY;
            const float x2 = (v1 && k0) ? sc[nt][2] * scale_log2 : -INFINITY;
            const float x3 = (v1 && k1) ? sc[nt][3] * scale_log2 : -INFINITY;
            float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
            }
            const float mn0 = fmaxf(m[nt][0], mx0), mn1 = fmaxf(m[nt][1], mx1);
            // a column that has seen no token yet keeps max -inf: exponentiate against 0
            const float ms0 = mn0 == -INFINITY ? 0.f : mn0, ms1 = mn1 == -INFINITY ? 0.f : mn1;
            const float al0 = ex2_approx(m[nt][0] - ms0), al1 = ex2_approx(m[nt][1] - ms1);
            m[nt][0] = mn0;
            m[nt][1] = mn1;
            const float e0 = ex2_approx(x0 - ms0), e1 = ex2_approx(x1 - ms1);
            const float e2 = ex2_approx(x2 - ms0), e3 = ex2_approx(x3 - ms1);
            const __nv_bfloat162 plo = __floats2bfloat162_rn(e0, e1);
            const __nv_bfloat162 phi = __floats2bfloat162_rn(e2, e3);
            float2 flo = __bfloat1622float2(plo), fhi = __bfloat1622float2(phi);
            if (split) {
                const __nv_bfloat162 rlo = __floats2bfloat162_rn(e0 - flo.x, e1 - flo.y);
                const __nv_bfloat162 rhi = __floats2bfloat162_rn(e2 - fhi.x, e3 - fhi.y);
                pl0[nt] = movmatrix_trans(*reinterpret_cast<const uint32_t *>(&rlo));
                pl1[nt] = movmatrix_trans(*reinterpret_cast<const uint32_t *>(&rhi));
                const float2 glo = __bfloat1622float2(rlo), ghi = __bfloat1622float2(rhi);
                flo.x += glo.x;
                flo.y += glo.y;
                fhi.x += ghi.x;
                fhi.y += ghi.y;
            }
            // the sum uses the rounded weights the PV product uses, so they stay normalised
            l[nt][0] = l[nt][0] * al0 + (flo.x + fhi.x);
            l[nt][1] = l[nt][1] * al1 + (flo.y + fhi.y);
#pragma unroll
            for (int mt = 0; mt < kSteps; ++mt) {
                acc[mt][nt][0] *= al0;
                acc[mt][nt][1] *= al1;
                acc[mt][nt][2] *= al0;
                acc[mt][nt][3] *= al1;
            }
            // P^T as the B operand of PV: transpose the (token x head) 8x8 quads
            pb0[nt] = movmatrix_trans(*reinterpret_cast<const uint32_t *>(&plo));
            pb1[nt] = movmatrix_trans(*reinterpret_cast<const uint32_t *>(&phi));
        }

#pragma unroll
        for (int mt = 0; mt < kSteps; ++mt) {
            const int u = mt >> 2;
            const int row = r8 + (mi >> 1) * 8;
            const int chunk = (mt & 3) * 2 + (mi & 1);
            uint32_t a[4];
            ldsm_x4_trans(sv + u * kSubBytes + row * 128 + ((chunk ^ (row & 7)) << 4), a);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(acc[mt][nt], a, pb0[nt], pb1[nt]);
            if (split) {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(acc[mt][nt], a, pl0[nt], pl1[nt]);
            }
        }
    }

    // Sums l over the 8 lanes that share each head column.
    __device__ __forceinline__ void reduce_l() {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int c = 0; c < 2; ++c)
#pragma unroll
                for (int o = 4; o < 32; o <<= 1) l[nt][c] += __shfl_xor_sync(0xffffffffu, l[nt][c], o);
    }
};

// =====================================================================================
// The per-block step for one query head per kv head (MHA, g = 1) on the CUDA
// cores. With a single query head the block's contraction is a matrix-vector
// product -- [16 tokens x D] . q and then [D x 16] . p -- that fills one of
// the tensor cores' eight MMA columns, so the warp does it in fp32 FMAs: the
// staged bf16 K and V are widened exactly to fp32 and the softmax weights stay
// fp32 (no rounding of p before P V). Same staged tiles, interface and state
// layout as WarpAttn, so the decode kernels take either.
//   scores: lane (quarter h4 = lane / 8, t8 = lane % 8) dots D/4 elements of
//     tokens t8 and t8 + 8 with the matching quarter of q; the four quarters
//     of a token are summed with two shuffles. Eight consecutive lanes read
//     eight different rows at one logical chunk, which the 128-byte swizzle
//     spreads over all banks.
//   softmax: m is kept equal in every lane; each lane of quarter 0 keeps the
//     running sum of its two tokens' weights (summed over lanes by reduce_l).
//   P V: lane owns output elements (D/32) lane .. + D/32 - 1; token t's
//     weight is broadcast from lane t % 8, its V row read 4 or 8 bytes a lane.
// =====================================================================================
template <int D>
struct WarpAttnScalar {
    static constexpr int kSubBytes = kBlock * 128;      // 2 KiB: 16 rows of 64 bf16
    static constexpr int kQuarter = D / 4;              // elements of a row one lane dots
    static constexpr int kChunks = kQuarter / 8;        // its 16-byte chunks (4 or 2)
    static constexpr int kWords = kQuarter / 2;         // its bf16 pairs (16 or 8)
    static constexpr int kDims = D / 32;                // output elements per lane (4 or 2)
    using QFrag = uint32_t[kWords];                     // the lane's quarter of q, bf16 pairs
    using Scores = float[2];                            // tokens t8 and t8 + 8
    float m, l;
    uint64_t acc[kDims / 2];                            // packed fp32 pairs: elements kDims*lane ..
    QFrag qw;                                           // widened to fp32 where used

    static __device__ __forceinline__ void load_q_frags(QFrag &f, const __nv_bfloat16 *q_group, int, int lane) {
        const uint4 *src = reinterpret_cast<const uint4 *>(q_group + (lane >> 3) * kQuarter);
#pragma unroll
        for (int j = 0; j < kChunks; ++j) {
            const uint4 v = __ldg(src + j);
            f[4 * j + 0] = v.x;
            f[4 * j + 1] = v.y;
            f[4 * j + 2] = v.z;
            f[4 * j + 3] = v.w;
        }
    }

    __device__ __forceinline__ void set_q(const QFrag &f) {
#pragma unroll
        for (int i = 0; i < kWords; ++i) qw[i] = f[i];
    }

    __device__ __forceinline__ void load_q(const __nv_bfloat16 *q_group, int g, int lane) {
        load_q_frags(qw, q_group, g, lane);
    }

    __device__ __forceinline__ void reset() {
        m = -INFINITY;
        l = 0.f;
#pragma unroll
        for (int i = 0; i < kDims / 2; ++i) acc[i] = 0;   // +0.0f, +0.0f
    }

    // s[p] = <q, K_t> for token t = t8 + 8 p of the staged K tile; each q pair
    // is widened once for both tokens.
    __device__ __forceinline__ void scores(uint32_t sk, Scores &s, int lane) const {
        const int h4 = lane >> 3, t8 = lane & 7;
        uint64_t a0 = 0, a1 = 0, b0 = 0, b1 = 0;        // token t8: a, token t8 + 8: b
#pragma unroll
        for (int j = 0; j < kChunks; ++j) {
            const int ci = h4 * kChunks + j;             // 16-byte chunk of the D-element row
            const int u = ci >> 3, c = ci & 7;           // 64-element sub-tile, chunk within its row
            const uint32_t at = sk + u * kSubBytes + ((c ^ t8) << 4);   // rows t8 and t8 + 8 share the swizzle
            uint32_t x[4], y[4];
            ld_shared_v4(at + t8 * 128, x);
            ld_shared_v4(at + (t8 + 8) * 128, y);
#pragma unroll
            for (int e = 0; e < 4; e += 2) {
                const uint64_t q0 = bf16x2_to_f2(qw[4 * j + e]), q1 = bf16x2_to_f2(qw[4 * j + e + 1]);
                a0 = fma_f2(bf16x2_to_f2(x[e]), q0, a0);
                a1 = fma_f2(bf16x2_to_f2(x[e + 1]), q1, a1);
                b0 = fma_f2(bf16x2_to_f2(y[e]), q0, b0);
                b1 = fma_f2(bf16x2_to_f2(y[e + 1]), q1, b1);
            }
        }
        float x0, x1, y0, y1;
        unpack_f2(add_f2(a0, a1), x0, x1);
        unpack_f2(add_f2(b0, b1), y0, y1);
        float d0 = x0 + x1, d1 = y0 + y1;
        d0 += __shfl_xor_sync(0xffffffffu, d0, 8);
        d1 += __shfl_xor_sync(0xffffffffu, d1, 8);
        d0 += __shfl_xor_sync(0xffffffffu, d0, 16);
        d1 += __shfl_xor_sync(0xffffffffu, d1, 16);
        s[0] = d0;
        s[1] = d1;
    }

    // Online-softmax update with the block's scores, then acc += V^T p.
    // Rows below `lo` are not tokens of the sequence (zero-filled by TMA).
    __device__ __forceinline__ void softmax_pv(const Scores &s, uint32_t sv, int lo, float scale_log2, int lane,
                                               int = 0, int = 0, bool = false) {
        const int h4 = lane >> 3, t8 = lane & 7;
        const float x0 = t8 >= lo ? s[0] * scale_log2 : -INFINITY;
        const float x1 = t8 + 8 >= lo ? s[1] * scale_log2 : -INFINITY;
        float mx = fmaxf(x0, x1);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        const float mn = fmaxf(m, mx);                   // finite: a block holds at least one token
        const float al = ex2_approx(m - mn);             // 0 on the first block (m = -inf)
        const float p0 = ex2_approx(x0 - mn), p1 = ex2_approx(x1 - mn);
        m = mn;
        l = l * al + (h4 == 0 ? p0 + p1 : 0.f);
        const uint64_t al2 = pack_f2(al, al);
        uint64_t a2[kDims / 2];                          // odd tokens in a second chain
#pragma unroll
        for (int i = 0; i < kDims / 2; ++i) {
            acc[i] = fma_f2(acc[i], al2, 0);
            a2[i] = 0;
        }
        // this lane's elements: 16-byte chunk ci of the row, at byte `off` in it
        constexpr int kLaneBytes = kDims * 2;
        const int ci = (lane * kLaneBytes) >> 4, off = (lane * kLaneBytes) & 15;
        const uint32_t vbase = sv + (ci >> 3) * kSubBytes + off;
        const int c = ci & 7;
        // two tokens per pass, even ones into acc and odd ones into a2; four
        // passes unrolled at a time keep the loads in flight without spilling
#pragma unroll 4
        for (int t = 0; t < kBlock; t += 2) {
            const float pe = __shfl_sync(0xffffffffu, t < 8 ? p0 : p1, t & 7);
            const float po = __shfl_sync(0xffffffffu, t < 8 ? p0 : p1, (t + 1) & 7);
            const uint64_t pe2 = pack_f2(pe, pe), po2 = pack_f2(po, po);
            const uint32_t ae = vbase + t * 128 + ((c ^ (t & 7)) << 4);
            const uint32_t ao = vbase + (t + 1) * 128 + ((c ^ ((t + 1) & 7)) << 4);
            if constexpr (kDims == 4) {
                uint32_t we[2], wo[2];
                ld_shared_v2(ae, we);
                ld_shared_v2(ao, wo);
                acc[0] = fma_f2(bf16x2_to_f2(we[0]), pe2, acc[0]);
                acc[1] = fma_f2(bf16x2_to_f2(we[1]), pe2, acc[1]);
                a2[0] = fma_f2(bf16x2_to_f2(wo[0]), po2, a2[0]);
                a2[1] = fma_f2(bf16x2_to_f2(wo[1]), po2, a2[1]);
            } else {
                uint32_t we, wo;
                asm volatile("ld.shared.b32 %0, [%1];" : "=r"(we) : "r"(ae));
                asm volatile("ld.shared.b32 %0, [%1];" : "=r"(wo) : "r"(ao));
                acc[0] = fma_f2(bf16x2_to_f2(we), pe2, acc[0]);
                a2[0] = fma_f2(bf16x2_to_f2(wo), po2, a2[0]);
            }
        }
#pragma unroll
        for (int i = 0; i < kDims / 2; ++i) acc[i] = add_f2(acc[i], a2[i]);
    }

    __device__ __forceinline__ void reduce_l() {
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    }

    template <typename OutT>
    __device__ __forceinline__ void store_rows(OutT *out_rows, int, int lane) const {
        const float inv = 1.f / l;
#pragma unroll
        for (int i = 0; i < kDims / 2; ++i) {
            float a, b;
            unpack_f2(acc[i], a, b);
            out_rows[kDims * lane + 2 * i] = to_out<OutT>(a * inv);
            out_rows[kDims * lane + 2 * i + 1] = to_out<OutT>(b * inv);
        }
    }

    __device__ __forceinline__ void block(uint32_t sk, uint32_t sv, int lo, float scale_log2, int lane, int = 0,
                                          int = 0, bool = false) {
        Scores sc;
        scores(sk, sc, lane);
        softmax_pv(sc, sv, lo, scale_log2, lane);
    }

    __device__ __forceinline__ void store_merge(float *ml, float *acc_rows, int, int lane) const {
        if (lane == 0) {
            ml[0] = m;
            ml[1] = l;
        }
#pragma unroll
        for (int i = 0; i < kDims / 2; ++i) {
            float a, b;
            unpack_f2(acc[i], a, b);
            acc_rows[kDims * lane + 2 * i] = a;
            acc_rows[kDims * lane + 2 * i + 1] = b;
        }
    }

    __device__ __forceinline__ void store_state(float *slot, int, int lane) const {
        if (lane == 0) {
            slot[0] = m;
            slot[1] = l;
        }
#pragma unroll
        for (int i = 0; i < kDims / 2; ++i) {
            float a, b;
            unpack_f2(acc[i], a, b);
            slot[2 + kDims * lane + 2 * i] = a;
            slot[2 + kDims * lane + 2 * i + 1] = b;
        }
    }
};

// =====================================================================================
// K1 (bf16, grid): one CTA per (split-context partition, kv head, sequence).
//
// Warp NCW is the producer: it reads the partition's block ids from the table
// 32 at a time and, for each block, issues TMA loads of the (block, kv head)
// K and V tiles -- [16 tokens][D] each, contiguous in HBM, one box each -- into a ring of
// NSTAGE shared-memory stages (128-byte swizzle, so fragment loads are free
// of bank conflicts). Warps 0..NCW-1 consume blocks round-robin, each with its
// own online-softmax state (WarpAttn). At the end the consumer warps merge
// their states through shared memory and either write the final output
// (single-partition sequence) or the partition's (max, sum, output) for the
// log-sum-exp reduce. Used for explicit partition sizes (and for batches
// larger than the persistent kernel's table of sequences).
// =====================================================================================
template <int D, int NT, int NSTAGE, int NCW>
struct Bf16Cfg {
    static constexpr int kSub = D / 64;                 // 128-byte-wide sub-tiles per tile
    static constexpr int kSubBytes = kBlock * 128;      // 2 KiB: 16 rows of 64 bf16
    static constexpr int kTile = kBlock * D * 2;        // one (block, head) tile of K or V
    static constexpr int kStage = 2 * kTile;            // K tile + V tile
    static constexpr int kSteps = D / 16;               // k-steps of QK^T, m-tiles of PV
    static constexpr int kThreads = (NCW + 1) * 32;
    static constexpr int kHeads = NT * 8;               // padded group width (MMA N)
    static constexpr int kMergeStride = D + 4;          // padded row of the merge buffer
    static constexpr int kMergeBytes = NCW * kHeads * (2 + kMergeStride) * 4;
    static constexpr int kBarOffset = NSTAGE * kStage;
    static constexpr int kSmem = kBarOffset + 2 * NSTAGE * 8 + 1024;  // + slack for 1 KiB alignment
    static_assert(kMergeBytes <= kBarOffset, "merge buffer must fit in the stage ring");
    static_assert(NSTAGE % NCW == 0, "each stage is always consumed by the same warp");
};

// Producer warp of the grid kernels: stages blocks [b0, b0 + nb) of one
// sequence's table row into the ring, 32 block ids at a time. `last_block` is
// the index of the sequence's last block and `last_valid` its token count
// (that block is loaded early so its slots past the end arrive zero-filled).
template <class C, int NSTAGE>
__device__ __forceinline__ void grid_produce(const CUtensorMap &tmk, const CUtensorMap &tmv, const int32_t *table_row,
                                             int b0, int nb, int last_block, int last_valid, int num_blocks,
                                             int num_kv_heads, int h, uint8_t *base, uint64_t *full, uint64_t *empty,
                                             int lane) {
    pdl_wait();  // the caches may have been written by the previous kernel (kv_append in a decode step)
    bool ok = true;
    for (int jb = 0; jb < nb && ok; jb += 32) {
        const int mine = (jb + lane < nb) ? __ldg(table_row + b0 + jb + lane) : 0;
        const int cnt = min(32, nb - jb);
        for (int i = 0; i < cnt; ++i) {
            const int pb = __shfl_sync(0xffffffffu, mine, i);
            const int j = jb + i;
            if (lane == 0) {
                const int st = j % NSTAGE;
                if (j >= NSTAGE && !mbar_wait(&empty[st], ((j / NSTAGE) - 1) & 1)) {
                    raise_error(PKV_DEVERR_TIMEOUT);
                    ok = false;
                }
                if (ok) {
                    int z;
                    if (pb < 0 || pb >= num_blocks) {
                        raise_error(PKV_DEVERR_BLOCK_ID);
                        z = -1;  // outside the tensor: the tile reads as zeros
                    } else {
                        z = pb * num_kv_heads + h;
                    }
                    const int y = (b0 + j == last_block) ? last_valid - kBlock : 0;
                    mbar_arrive_expect_tx(&full[st], C::kStage);
                    uint8_t *sk = base + st * C::kStage;
                    tma_load_4d_hint(sk, &tmk, 0, y, 0, z, &full[st], l2_evict_first());
                    tma_load_4d_hint(sk + C::kTile, &tmv, 0, y, 0, z, &full[st], l2_evict_first());
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
        }
    }
}

// Consumer warps of the grid kernels: blocks j = warp, warp + NCW, ... of the
// staged range (block_args(j, stage) gives each block's early-loaded rows and
// column range), then the warps' states merged through shared memory. For
// each column c < ncols (an MMA column: a query head of a query sequence)
// and head-dim index d, emit(c, d, o, M, L) receives the column's output
// o = O / L and its (max, sum) in the log2 domain.
template <class C, int D, int NSTAGE, int NCW, class WA, class BlockArgs, class Emit>
__device__ __forceinline__ void grid_consume(WA &wa, int nb, BlockArgs block_args, float scale_log2, uint8_t *base,
                                             uint64_t *full, uint64_t *empty, int ncols, int warp, int lane, int tid,
                                             Emit emit) {
    for (int j = warp; j < nb; j += NCW) {
        const int st = j % NSTAGE;
        if (!mbar_wait(&full[st], (j / NSTAGE) & 1)) {
            raise_error(PKV_DEVERR_TIMEOUT);
            break;
        }
        const uint32_t sk = smem_u32(base + st * C::kStage);
        const int4 a = block_args(j, st);  // (rows loaded early, first column, column end, split)
        wa.block(sk, sk + C::kTile, a.x, scale_log2, lane, a.y, a.z, a.w != 0);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
    }
    wa.reduce_l();
    named_barrier_sync(1, NCW * 32);  // every consumer is done with the stage ring
    float *mml = reinterpret_cast<float *>(base);                    // [NCW][kHeads][2]
    float *macc = mml + NCW * C::kHeads * 2;                         // [NCW][kHeads][kMergeStride]
    wa.store_merge(mml + warp * C::kHeads * 2, macc + warp * C::kHeads * C::kMergeStride, C::kMergeStride, lane);
    named_barrier_sync(1, NCW * 32);
    for (int idx = tid; idx < ncols * D; idx += NCW * 32) {
        const int col = idx / D, d = idx - col * D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NCW; ++w) M = fmaxf(M, mml[(w * C::kHeads + col) * 2]);
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < NCW; ++w) {
            const float mw = mml[(w * C::kHeads + col) * 2];
            const float f = (mw == -INFINITY) ? 0.f : ex2_approx(mw - M);
            L += mml[(w * C::kHeads + col) * 2 + 1] * f;
            O += macc[(w * C::kHeads + col) * C::kMergeStride + d] * f;
        }
        emit(col, d, O / L, M, L);
    }
}

template <int D, int NT, int NSTAGE, int NCW, typename OutT = __nv_bfloat16, class WA = WarpAttn<D, NT>>
__global__ void __launch_bounds__((NCW + 1) * 32)
    decode_bf16_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                       const DecodeParams p) {
    using C = Bf16Cfg<D, NT, NSTAGE, NCW>;
    extern __shared__ uint8_t smem_raw[];

    const int part = blockIdx.x, h = blockIdx.y, s = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = p.group;
    const int len = seq_len(p, s, tid == 0 && part == 0 && h == 0);
    const int nblk = (len + kBlock - 1) / kBlock;
    const int npart = (nblk + p.part_blocks - 1) / p.part_blocks;
    OutT *out = static_cast<OutT *>(p.out);

    if (len == 0) {  // empty context: zero output rows
        if (part == 0) {
            OutT *o = out + ((size_t)s * p.num_q_heads + (size_t)h * g) * D;
            for (int i = tid; i < g * D; i += C::kThreads) o[i] = to_out<OutT>(0.f);
        }
        return;
    }
    if (part >= npart) return;

    const int b_begin = part * p.part_blocks;
    const int nb = min(nblk - b_begin, p.part_blocks);
    const int last_valid = len - (nblk - 1) * kBlock;  // tokens in the sequence's last block

    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(base + C::kBarOffset);
    uint64_t *empty = full + NSTAGE;
    if (tid == 0) {
        prefetch_tensormap(&tmk);
        prefetch_tensormap(&tmv);
        for (int i = 0; i < NSTAGE; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        mbar_fence_init();
    }
    __syncthreads();

    if (warp == NCW) {
        grid_produce<C, NSTAGE>(tmk, tmv, p.block_tables + (size_t)s * p.max_blocks_per_seq, b_begin, nb, nblk - 1,
                                last_valid, p.num_blocks, p.num_kv_heads, h, base, full, empty, lane);
        return;
    }
    WA wa;
    wa.load_q(static_cast<const __nv_bfloat16 *>(p.q) + ((size_t)s * p.num_q_heads + (size_t)h * g) * D, g, lane);
    wa.reset();
    const size_t orow0 = (size_t)s * p.num_q_heads + (size_t)h * g;
    const int last_in_range = (b_begin + nb - 1 == nblk - 1) ? nb - 1 : -1;
    grid_consume<C, D, NSTAGE, NCW>(
        wa, nb,
        [&](int j, int) {
            return make_int4(j == last_in_range ? kBlock - last_valid : 0, 0, C::kHeads, b_begin + j < kSplitBlocks);
        },
        p.scale_log2, base, full, empty, g, warp, lane, tid, [&](int col, int d, float o, float M, float L) {
            if (npart == 1) {
                out[(orow0 + col) * D + d] = to_out<OutT>(o);
            } else {
                const size_t r = (orow0 + col) * p.max_parts + part;
                p.ws_o[r * D + d] = o;
                if (d == 0) {
                    p.ws_ml[r * 2 + 0] = M;
                    p.ws_ml[r * 2 + 1] = L;
                }
            }
        });
}

// =====================================================================================
// K1 (bf16, persistent): one CTA per SM, NW warps, each warp an independent
// decode worker with its own NS-stage TMA ring.
//
// All (sequence, kv head) units' blocks form one sequence of positions
// (sequence-major, then head, then block); the T positions are cut into W
// equal ranges, one per warp, so every warp streams the same number of K/V
// tiles whatever the length mix. A warp walks its range block by block --
// lane 0 keeps the ring NS blocks ahead with TMA, the lanes gather the block
// ids of the next 32 positions ahead of use -- and keeps one online-softmax
// state per unit segment. A unit that lies inside one range is written out
// directly. A unit cut by range boundaries leaves one (max, sum, acc) state
// per segment in the workspace; the warp that finishes the unit's last
// outstanding segment (an arrival counter per cut unit, kept at the head of
// the workspace, where no other decode path writes) merges the segments with
// the log-sum-exp rule in segment order and writes the output, so the result
// does not depend on which warp arrives last.
// =====================================================================================
template <int D, int NT, int NS, int NW>
struct PersistCfg {
    static constexpr int kSub = D / 64;
    static constexpr int kSubBytes = kBlock * 128;
    static constexpr int kTile = kBlock * D * 2;
    static constexpr int kStage = 2 * kTile;
    static constexpr int kSteps = D / 16;
    static constexpr int kThreads = NW * 32;
    static constexpr int kRing = NW * NS * kStage;
    static constexpr int kBarOffset = kRing;                         // K-full then V-full barriers
    static constexpr int kPrefixOffset = kBarOffset + 2 * NW * NS * 8;
    static constexpr size_t smem_bytes(int num_seqs) { return kPrefixOffset + (size_t)(num_seqs + 1) * 4 + 1024; }
};

// Position cursor: sequence s (with n = its blocks), kv head h, block j.
struct Cursor {
    int s, h, j, n;
};

// Moves c forward by k >= 0 positions; prefix[] holds the block-count prefix
// sums. The caller guarantees the target position exists.
__device__ __forceinline__ void cursor_advance(Cursor &c, int k, const int *prefix, int num_kv_heads) {
    while (c.j + k >= c.n) {
        k -= c.n - c.j;
        c.j = 0;
        if (++c.h == num_kv_heads) {
            c.h = 0;
            do {
                ++c.s;
                c.n = prefix[c.s + 1] - prefix[c.s];
            } while (c.n == 0);
        }
    }
    c.j += k;
}

// Merges the nseg segment states of one cut unit (worker w1's second slot,
// then the first slots of workers w1+1 ..) with the log-sum-exp rule and
// writes the g output rows. One warp; lane k holds segment k's weights, and
// every lane accumulates head-dim elements lane, lane+32, .. of all heads
// with the loads of two segments in flight at a time.
template <int D, typename OutT>
__device__ __forceinline__ void merge_segments(const float *partials, size_t slot_floats, int w1, int nseg, int g,
                                               OutT *out_rows, int lane) {
    constexpr int PER = D / 32;
    auto seg_row = [&](int k, int head) -> const float * {
        return partials + (size_t)(2 * (w1 + k) + (k == 0 ? 1 : 0)) * slot_floats + (size_t)head * (2 + D);
    };
    for (int head = 0; head < g; ++head) {
        // M and L over all segments, 32 segments per pass
        float M = -INFINITY;
        for (int k0 = 0; k0 < nseg; k0 += 32) {
            const float mk = (k0 + lane < nseg) ? __ldcg(seg_row(k0 + lane, head)) : -INFINITY;
            M = fmaxf(M, mk);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        float L = 0.f;
        for (int k0 = 0; k0 < nseg; k0 += 32) {
            const int k = k0 + lane;
            if (k < nseg) {
                const float *r = seg_row(k, head);
                const float mk = __ldcg(r);
                if (mk != -INFINITY) L += __ldcg(r + 1) * ex2_approx(mk - M);
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
        const float invL = 1.f / L;
        float acc[PER];
#pragma unroll
        for (int i = 0; i < PER; ++i) acc[i] = 0.f;
        for (int k0 = 0; k0 < nseg; k0 += 32) {
            const int kk = k0 + lane;
            float ck = 0.f;
            if (kk < nseg) {
                const float mk = __ldcg(seg_row(kk, head));
                ck = (mk == -INFINITY) ? 0.f : ex2_approx(mk - M) * invL;
            }
            const int nk = min(32, nseg - k0);
            int k = 0;
            for (; k + 2 <= nk; k += 2) {
                const float c0 = __shfl_sync(0xffffffffu, ck, k), c1 = __shfl_sync(0xffffffffu, ck, k + 1);
                const float *r0 = seg_row(k0 + k, head) + 2, *r1 = seg_row(k0 + k + 1, head) + 2;
                float v0[PER], v1[PER];
#pragma unroll
                for (int i = 0; i < PER; ++i) {
                    v0[i] = __ldcg(r0 + lane + 32 * i);
                    v1[i] = __ldcg(r1 + lane + 32 * i);
                }
#pragma unroll
                for (int i = 0; i < PER; ++i) acc[i] = fmaf(c0, v0[i], fmaf(c1, v1[i], acc[i]));
            }
            for (; k < nk; ++k) {
                const float c0 = __shfl_sync(0xffffffffu, ck, k);
                const float *r0 = seg_row(k0 + k, head) + 2;
#pragma unroll
                for (int i = 0; i < PER; ++i) acc[i] = fmaf(c0, __ldcg(r0 + lane + 32 * i), acc[i]);
            }
        }
#pragma unroll
        for (int i = 0; i < PER; ++i) out_rows[(size_t)head * D + lane + 32 * i] = to_out<OutT>(acc[i]);
    }
}

// WA: the per-block step -- WarpAttn (tensor cores, any group up to 8 NT) or
// WarpAttnScalar (CUDA cores, one query head per kv head).
template <int D, int NT, int NS, int NW, typename OutT = __nv_bfloat16, class WA = WarpAttn<D, NT>>
__global__ void __launch_bounds__(NW * 32, 1)
    decode_bf16_persistent_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                                  const DecodeParams p) {
    using C = PersistCfg<D, NT, NS, NW>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ int warp_total[NW];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int S = p.num_seqs, Hkv = p.num_kv_heads, g = p.group;
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(base + C::kBarOffset);
    int *prefix = reinterpret_cast<int *>(base + C::kPrefixOffset);
    OutT *out = static_cast<OutT *>(p.out);

    if (tid == 0) {
        prefetch_tensormap(&tmk);
        prefetch_tensormap(&tmv);
        for (int i = 0; i < 2 * NW * NS; ++i) mbar_init(&full[i], 1);
        mbar_fence_init();
    }

    // ---- block-count prefix sums over the batch (every CTA computes its own copy) ----
    const int per = (S + C::kThreads - 1) / C::kThreads;
    const int s_lo = min(S, tid * per), s_hi = min(S, s_lo + per);
    int local = 0;
    for (int s = s_lo; s < s_hi; ++s) local += (seq_len(p, s, blockIdx.x == 0) + kBlock - 1) / kBlock;
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) warp_total[warp] = incl;
    __syncthreads();
    int run = incl - local;
    for (int w = 0; w < warp; ++w) run += warp_total[w];
    for (int s = s_lo; s < s_hi; ++s) {
        prefix[s] = run;
        run += (seq_len(p, s, false) + kBlock - 1) / kBlock;
    }
    if (tid == 0) {
        int tot = 0;
        for (int w = 0; w < NW; ++w) tot += warp_total[w];
        prefix[S] = tot;
    }
    __syncthreads();

    // ---- empty contexts: zero output rows (spread over the CTAs) ----
    for (int s = blockIdx.x; s < S; s += gridDim.x) {
        if (prefix[s + 1] == prefix[s]) {
            OutT *o = out + (size_t)s * p.num_q_heads * D;
            for (int i = tid; i < p.num_q_heads * D; i += C::kThreads) o[i] = to_out<OutT>(0.f);
        }
    }

    // ---- this warp's range of positions ----
    // W = min(warps, T) workers, so every worker's range is non-empty and the
    // workers covering a unit are consecutive
    const long long T = (long long)Hkv * prefix[S];
    const int W = (int)min((long long)gridDim.x * NW, T);
    const int w = blockIdx.x * NW + warp;
    if (w >= W) return;
    const long long start = T * w / W, end = T * (w + 1) / W;
    const int cnt = (int)(end - start);

    Cursor c;
    {
        int lo = 0, hi = S - 1;  // largest s with Hkv * prefix[s] <= start (never an empty sequence)
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if ((long long)Hkv * prefix[mid] <= start) lo = mid; else hi = mid - 1;
        }
        c.s = lo;
        c.n = prefix[lo + 1] - prefix[lo];
        const int r = (int)(start - (long long)Hkv * prefix[lo]);
        c.h = r / c.n;
        c.j = r - c.h * c.n;
    }

    // Block ids of the 32 positions starting at cursor b (lane i: position b + i),
    // and beside each, 16 * kv head + the rows its tile starts early (16 - valid
    // tokens on a sequence's last block, else 0). Nothing here waits on the
    // loads: they are checked when the position is issued, 32 blocks later.
    struct Batch {
        int pb, hs;
    };
    auto batch_of = [&](Cursor b, int count) -> Batch {
        Batch r{0, 0};
        if (lane < count) {
            cursor_advance(b, lane, prefix, Hkv);
            r.pb = __ldg(p.block_tables + (size_t)b.s * p.max_blocks_per_seq + b.j);
            const int shift = (b.j == b.n - 1) ? kBlock * b.n - seq_len(p, b.s, false) : 0;
            r.hs = b.h * 16 + shift;
        }
        return r;
    };

    uint64_t *kfull = full + warp * NS;
    uint64_t *vfull = full + NW * NS + warp * NS;
    uint8_t *ring = base + warp * NS * C::kStage;
    Cursor bnext = c;
    Batch cur = batch_of(c, min(32, cnt));
    Batch nxt{0, 0};
    if (cnt > 32) {
        cursor_advance(bnext, 32, prefix, Hkv);
        nxt = batch_of(bnext, min(32, cnt - 32));
    }
    // K and V of block b are issued separately (K first), both by lane 0.
    int kissued = 0, vissued = 0;
    int z_last = 0, y_last = 0;  // coordinates of the last K issued, reused by its V
    auto issue_k = [&]() {
        if (kissued > 0 && (kissued & 31) == 0) {
            cur = nxt;
            if (kissued + 32 < cnt) {
                cursor_advance(bnext, 32, prefix, Hkv);
                nxt = batch_of(bnext, min(32, cnt - kissued - 32));
            }
        }
        const int pb = __shfl_sync(0xffffffffu, cur.pb, kissued & 31);
        const int hs = __shfl_sync(0xffffffffu, cur.hs, kissued & 31);
        if (lane == 0) {
            if (pb < 0 || pb >= p.num_blocks) {
                raise_error(PKV_DEVERR_BLOCK_ID);
                z_last = -1;  // outside the tensor: the tile reads as zeros
            } else {
                z_last = pb * Hkv + (hs >> 4);
            }
            y_last = -(hs & 15);
            const int st = kissued % NS;
            mbar_arrive_expect_tx(&kfull[st], C::kTile);
            uint8_t *sk = ring + st * C::kStage;
            tma_load_4d_hint(sk, &tmk, 0, y_last, 0, z_last, &kfull[st], l2_evict_first());
        }
        ++kissued;
    };
    auto issue_v = [&]() {
        if (lane == 0) {
            const int st = vissued % NS;
            mbar_arrive_expect_tx(&vfull[st], C::kTile);
            uint8_t *sv = ring + st * C::kStage + C::kTile;
            tma_load_4d_hint(sv, &tmv, 0, y_last, 0, z_last, &vfull[st], l2_evict_first());
        }
        ++vissued;
    };
    pdl_wait();  // the caches may have been written by the previous kernel (kv_append in a decode step)
    while (kissued < min(NS, cnt)) {
        issue_k();
        issue_v();
    }

    const size_t slot_floats = (size_t)g * (2 + D);
    WA wa;
    int seg_j0 = c.j;
    int len = seq_len(p, c.s, false);
    wa.load_q(static_cast<const __nv_bfloat16 *>(p.q) + ((size_t)c.s * p.num_q_heads + (size_t)c.h * g) * D, g, lane);
    wa.reset();

    const __nv_bfloat16 *qbase = static_cast<const __nv_bfloat16 *>(p.q);
    typename WA::QFrag qnext;
    int len_next = 0;
    for (int i = 0; i < cnt; ++i) {
        const int st = i % NS;
        const bool unit_end = c.j == c.n - 1;
        Cursor cn = c;
        if (unit_end && i != cnt - 1) {
            // the next unit's query and length, in flight while this block computes
            cursor_advance(cn, 1, prefix, Hkv);
            WA::load_q_frags(qnext, qbase + ((size_t)cn.s * p.num_q_heads + (size_t)cn.h * g) * D, g, lane);
            len_next = seq_len(p, cn.s, false);
        }
        const uint32_t sk = smem_u32(ring + st * C::kStage);
        const uint32_t par = (i / NS) & 1;
        if (!mbar_wait(&kfull[st], par)) {
            raise_error(PKV_DEVERR_TIMEOUT);
            break;
        }
        typename WA::Scores sc;
        wa.scores(sk, sc, lane);
        __syncwarp();  // every lane's K fragment loads are done before the K refill
        const bool refill = kissued < cnt;
        if (refill) issue_k();
        if (!mbar_wait(&vfull[st], par)) {
            raise_error(PKV_DEVERR_TIMEOUT);
            break;
        }
        wa.softmax_pv(sc, sk + C::kTile, unit_end ? kBlock * c.n - len : 0, p.scale_log2, lane, 0, 8 * NT,
                      c.j < kSplitBlocks);
        __syncwarp();  // ... and its V fragment loads before the V refill
        if (refill) issue_v();

        if (!unit_end && i != cnt - 1) {
            ++c.j;
            continue;
        }
        // ---- the segment ends here ----
        wa.reduce_l();
        const size_t orow0 = (size_t)c.s * p.num_q_heads + (size_t)c.h * g;
        if (seg_j0 == 0 && unit_end) {
            // the whole unit: write the output from the registers
            wa.store_rows(out + orow0 * D, g, lane);
        } else {
            // a cut unit: leave this segment's state, then the last arrival merges
            wa.store_state(p.partials + (size_t)(2 * w + (seg_j0 == 0 ? 1 : 0)) * slot_floats, g, lane);
            __syncwarp();  // every lane's state writes are ordered before lane 0's release below
            // workers w1..w2 cover the unit; w1 (the worker holding its first
            // position) is the first worker of no other cut unit -- only one
            // unit spans the end of a worker's range -- so counters[w1] is
            // this unit's own arrival counter
            const long long x0 = (long long)Hkv * prefix[c.s] + (long long)c.h * c.n;
            const int w1 = (int)(((x0 + 1) * W - 1) / T);
            const int w2 = (int)(((x0 + c.n) * W - 1) / T);
            int prev = 0;
            if (lane == 0) prev = atomic_add_acq_rel_gpu(p.counters + w1, 1);
            prev = __shfl_sync(0xffffffffu, prev, 0);
            if (prev == w2 - w1) {
                __syncwarp();  // lane 0's acquire covers the lanes reading the other segments
                merge_segments<D, OutT>(p.partials, slot_floats, w1, w2 - w1 + 1, g, out + orow0 * D, lane);
                if (lane == 0) p.counters[w1] = 0;  // ready for the next call
            }
        }
        if (i == cnt - 1) break;
        // ---- next unit ----
        c = cn;
        seg_j0 = 0;
        len = len_next;
        wa.set_q(qnext);
        wa.reset();
    }
}

// =====================================================================================
// K1 (bf16, shared prefix): decode for batches whose sequences share leading
// blocks -- parallel samples of one prompt, a common system prompt
// ("Batching Continuo y PagedAttention", cruxr.ai, copy-on-write paragraph:
// the tables of requests with a common prefix point at the same physical
// blocks). A unit is a group and a kv head; its blocks are the union of the
// members' contexts: the shared prefix once (read through the first member's
// table), then each member's own blocks. All members' query heads are the
// MMA columns (member m, head n = column m * g + n); a prefix block is
// attended for every column, a member's own block for that member's columns
// only, so each column's online softmax covers exactly its sequence's
// context and each shared block is read from HBM once per group. Sequences in
// no group are listed as groups of one. grid (partition, kv head, group).
// Every partition leaves a (max, sum, output) state per column;
// cascade_reduce_kernel merges a row's states with the log-sum-exp rule.
// =====================================================================================
constexpr int kMaxGroup = 16;

struct UnionUnit {
    int count;                   // members (valid ones, in slot order)
    int prefix;                  // shared blocks, read through member 0's table
    int total;                   // blocks in the union
    int member[kMaxGroup];       // sequence ids
    int len[kMaxGroup];          // their context lengths
    int own[kMaxGroup + 1];      // union position where each member's own blocks start
};

// Builds group z's union unit in shared memory with one warp (lane m reads
// member slot m): members in slot order, the blocks they share (cut to the
// shortest member's full blocks), and where each member's own blocks start.
__device__ __forceinline__ void union_unit(const DecodeParams &p, int z, UnionUnit &u, int lane, bool flag) {
    const int M = p.group_size;
    int sm = -1, len = 0;
    if (lane < M) {
        sm = __ldg(p.group_members + (size_t)z * M + lane);
        if (sm < 0 || sm >= p.num_seqs) sm = -1;
        else len = seq_len(p, sm, flag);
    }
    const unsigned valid = __ballot_sync(0xffffffffu, sm >= 0);
    int pb = sm >= 0 ? len / kBlock : INT_MAX;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) pb = min(pb, __shfl_xor_sync(0xffffffffu, pb, o));
    const int shared = valid ? min(pb, max(__ldg(p.shared_blocks + z), 0)) : 0;
    const int idx = __popc(valid & ((1u << lane) - 1));   // this member's place among the valid ones
    const int own = sm >= 0 ? (len + kBlock - 1) / kBlock - shared : 0;
    int incl = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (sm >= 0) {
        u.member[idx] = sm;
        u.len[idx] = len;
        u.own[idx] = shared + incl - own;
    }
    if (lane == 31) {
        u.count = __popc(valid);
        u.prefix = shared;
        u.total = shared + incl;
        u.own[__popc(valid)] = shared + incl;
    }
}

template <int D, int NT, int NSTAGE, int NCW>
__global__ void __launch_bounds__((NCW + 1) * 32)
    decode_bf16_cascade_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                               const DecodeParams p) {
    using C = Bf16Cfg<D, NT, NSTAGE, NCW>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ UnionUnit u;
    __shared__ int2 stage_info[NSTAGE];  // per stage: (member or -1 for the prefix, rows loaded early | split << 8)

    const int part = blockIdx.x, h = blockIdx.y, z = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = p.group;
    if (warp == 0) union_unit(p, z, u, lane, part == 0 && h == 0);
    __syncthreads();
    if (part == 0 && h == 0 && tid == 0)  // for the reduce: how many partitions the group's rows have
        p.counters[z] = u.count ? (u.total + p.part_blocks - 1) / p.part_blocks : 0;
    const int j0 = part * p.part_blocks;
    if (u.count == 0 || j0 >= u.total) return;
    const int nb = min(u.total - j0, p.part_blocks);

    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(base + C::kBarOffset);
    uint64_t *empty = full + NSTAGE;
    if (tid == 0) {
        prefetch_tensormap(&tmk);
        prefetch_tensormap(&tmv);
        for (int i = 0; i < NSTAGE; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        mbar_fence_init();
    }
    __syncthreads();

    if (warp == NCW) {
        // ------------------------------ producer ------------------------------
        bool ok = true;
        for (int jb = 0; jb < nb && ok; jb += 32) {
            int pb = 0, mem = -1, early = 0;
            if (jb + lane < nb) {
                const int j = j0 + jb + lane;
                int row = u.member[0], blk = j;
                if (j >= u.prefix) {
                    mem = 0;
                    while (j >= u.own[mem + 1]) ++mem;
                    row = u.member[mem];
                    blk = u.prefix + (j - u.own[mem]);
                    const int nblk = (u.len[mem] + kBlock - 1) / kBlock;
                    if (blk == nblk - 1) early = kBlock * nblk - u.len[mem];
                }
                pb = __ldg(p.block_tables + (size_t)row * p.max_blocks_per_seq + blk);
                if (blk < kSplitBlocks) early |= 1 << 8;  // the consumers' split flag rides above the row count
            }
            const int cnt = min(32, nb - jb);
            for (int i = 0; i < cnt; ++i) {
                const int bpb = __shfl_sync(0xffffffffu, pb, i);
                const int bmem = __shfl_sync(0xffffffffu, mem, i);
                const int bearly = __shfl_sync(0xffffffffu, early, i);
                const int jj = jb + i;
                if (lane == 0) {
                    const int st = jj % NSTAGE;
                    if (jj >= NSTAGE && !mbar_wait(&empty[st], ((jj / NSTAGE) - 1) & 1)) {
                        raise_error(PKV_DEVERR_TIMEOUT);
                        ok = false;
                    }
                    if (ok) {
                        int zt;
                        if (bpb < 0 || bpb >= p.num_blocks) {
                            raise_error(PKV_DEVERR_BLOCK_ID);
                            zt = -1;
                        } else {
                            zt = bpb * p.num_kv_heads + h;
                        }
                        stage_info[st] = make_int2(bmem, bearly);
                        mbar_arrive_expect_tx(&full[st], C::kStage);
                        uint8_t *sk = base + st * C::kStage;
                        tma_load_4d_hint(sk, &tmk, 0, -(bearly & 0xff), 0, zt, &full[st], l2_evict_first());
                        tma_load_4d_hint(sk + C::kTile, &tmv, 0, -(bearly & 0xff), 0, zt, &full[st], l2_evict_first());
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
            }
        }
        return;
    }
    // output row (sequence * Hq + query head) of each MMA column, -1 if unused
    auto row_of = [&](int col) -> int {
        const int m = col / g;
        return m < u.count ? u.member[m] * p.num_q_heads + h * g + (col - m * g) : -1;
    };
    WarpAttn<D, NT> wa;
    wa.load_q_rows(static_cast<const __nv_bfloat16 *>(p.q), row_of, lane);
    wa.reset();
    const int ncols = min(u.count * g, C::kHeads);
    grid_consume<C, D, NSTAGE, NCW>(
        wa, nb,
        [&](int, int st) {
            const int2 info = stage_info[st];
            const int early = info.y & 0xff, split = info.y >> 8;
            return info.x < 0 ? make_int4(early, 0, ncols, split) : make_int4(early, info.x * g, info.x * g + g, split);
        },
        p.scale_log2, base, full, empty, ncols, warp, lane, tid, [&](int col, int d, float o, float Mx, float L) {
            const int r0 = row_of(col);
            if (r0 < 0) return;
            const size_t r = (size_t)r0 * p.max_parts + part;
            p.ws_o[r * D + d] = L > 0.f ? o : 0.f;  // a column this partition never attended leaves an empty state
            if (d == 0) {
                p.ws_ml[r * 2 + 0] = Mx;
                p.ws_ml[r * 2 + 1] = L;
            }
        });
}

// Merges each (sequence, query head) row's partition states (log-sum-exp
// rule, empty states skipped); a row with none gives zeros. One warp per
// (group, member slot, query head): lane k holds partition k's (max, sum),
// every lane accumulates head-dim elements lane, lane + 32, .., with the
// partition outputs of up to kReduceBatch partitions in flight at a time.
constexpr int kReduceWarps = 8, kReduceBatch = 8;
template <int D>
__global__ void __launch_bounds__(kReduceWarps * 32) cascade_reduce_kernel(const DecodeParams p) {
    constexpr int PER = D / 32;
    const int lane = threadIdx.x & 31, Hq = p.num_q_heads, M = p.group_size;
    const long long r = (long long)blockIdx.x * kReduceWarps + (threadIdx.x >> 5);
    if (r >= (long long)p.num_groups * M * Hq) return;
    const int hq = (int)(r % Hq);
    const long long zm = r / Hq;
    const int m = (int)(zm % M), z = (int)(zm / M);
    const int s = __ldg(p.group_members + (size_t)z * M + m);
    const int n = __ldcg(p.counters + z);  // the group's partitions (written by the shared-prefix kernel)
    if (s < 0 || s >= p.num_seqs) return;
    const size_t row = (size_t)s * Hq + hq;
    __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(p.out) + row * D;
    const float *ml = p.ws_ml + row * p.max_parts * 2;
    const float *o = p.ws_o + row * p.max_parts * D;
    // the row's max and weight sum over all partitions, 32 per pass
    float Mx = -INFINITY, W = 0.f;
    for (int k0 = 0; k0 < n; k0 += 32) {
        float mk = -INFINITY, lk = 0.f;
        if (k0 + lane < n) {
            const float2 v = __ldcg(reinterpret_cast<const float2 *>(ml) + k0 + lane);
            mk = v.x;
            lk = v.y;
        }
        float Mp = mk;
#pragma unroll
        for (int sh = 16; sh > 0; sh >>= 1) Mp = fmaxf(Mp, __shfl_xor_sync(0xffffffffu, Mp, sh));
        float Wp = mk == -INFINITY ? 0.f : lk * exp2f(mk - Mp);
#pragma unroll
        for (int sh = 16; sh > 0; sh >>= 1) Wp += __shfl_xor_sync(0xffffffffu, Wp, sh);
        const float Mn = fmaxf(Mx, Mp);
        W = (Mx == -INFINITY ? 0.f : W * exp2f(Mx - Mn)) + (Mp == -INFINITY ? 0.f : Wp * exp2f(Mp - Mn));
        Mx = Mn;
    }
    if (Mx == -INFINITY) {  // nothing attended: empty context
#pragma unroll
        for (int i = 0; i < PER; ++i) out[lane + 32 * i] = __float2bfloat16_rn(0.f);
        return;
    }
    const float invW = 1.f / W;
    float acc[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) acc[i] = 0.f;
    float ck = 0.f;  // lane k: the weight of partition (32-block base) + k
    for (int k0 = 0; k0 < n; k0 += kReduceBatch) {
        if ((k0 & 31) == 0) {
            const int k = k0 + lane;
            ck = 0.f;
            if (k < n) {
                const float2 v = __ldcg(reinterpret_cast<const float2 *>(ml) + k);
                ck = v.x == -INFINITY ? 0.f : v.y * exp2f(v.x - Mx) * invW;
            }
        }
        float vals[kReduceBatch][PER];
#pragma unroll
        for (int b = 0; b < kReduceBatch; ++b)
#pragma unroll
            for (int i = 0; i < PER; ++i) vals[b][i] = k0 + b < n ? __ldcg(o + (size_t)(k0 + b) * D + lane + 32 * i) : 0.f;
#pragma unroll
        for (int b = 0; b < kReduceBatch; ++b) {
            const float c = __shfl_sync(0xffffffffu, ck, (k0 + b) & 31);
#pragma unroll
            for (int i = 0; i < PER; ++i) acc[i] = fmaf(c, vals[b][i], acc[i]);
        }
    }
#pragma unroll
    for (int i = 0; i < PER; ++i) out[lane + 32 * i] = __float2bfloat16_rn(acc[i]);
}

// Prefill (bf16) parameters: causal attention for several new tokens per
// sequence (the kernel is in pkv_prefill_tc.cuh).
struct PrefillParams {
    DecodeParams d;
    const int32_t *query_start;  // [S + 1]
    int tile_tokens;             // query tokens per 128-row tile (128 / g)
    int max_query_len;           // the grid covers this many new tokens per sequence
    int num_queries;             // rows of q and out
    int seq_major;               // CTA order: one sequence at a time (1) or pair index slowest (0)
};

// =====================================================================================
// K1 (fp32, staged): the grid kernel's decomposition for fp32 caches. Warp NCW stages
// each (block, kv head) K and V tile -- [16 tokens][D] fp32, contiguous in HBM -- by TMA
// into an NSTAGE ring, as D / 32 sub-tiles of 16 rows x 128 bytes with the 128-byte
// swizzle; warps 0..NCW-1 (alone, or in teams of two that split a block's query heads)
// run WarpAttnF32 on the CUDA cores over their blocks and merge their states through
// shared memory. The group's query rows are staged in shared memory once per CTA.
// =====================================================================================
// Query-head bound from which two warps share each block (each half the heads).
#ifndef PKV_F32_SPLIT_FROM
#define PKV_F32_SPLIT_FROM 4
#endif

template <int D, int GMAX, int NSTAGE, int NCW>
struct F32Cfg {
    static constexpr int kTile = kBlock * D * 4;                 // one (block, head) tile of K or V
    static constexpr int kStage = 2 * kTile;                     // K tile + V tile
    static constexpr int kThreads = (NCW + 1) * 32;
    static constexpr int kSplit = GMAX >= PKV_F32_SPLIT_FROM ? 2 : 1;  // warps sharing a block (each half the heads)
    static constexpr int kTeams = NCW / kSplit;
    static constexpr int kWarpHeads = GMAX / kSplit;             // query-head bound of one warp
    static constexpr int kMergeStride = D + 4;
    static constexpr int kMergeBytes = NCW * kWarpHeads * (2 + kMergeStride) * 4;
    static constexpr int kQuarterBytes = D + 16;                 // a quarter row of q (D / 4 fp32) + 16 bytes
    static constexpr int kQRow = 4 * kQuarterBytes;
    static constexpr int kPBytes = kWarpHeads * kBlock * 4;      // one warp's weights of a block
    static constexpr int kBarOffset = NSTAGE * kStage;
    static constexpr int kQOffset = kBarOffset + 2 * NSTAGE * 8;
    static constexpr int kPOffset = kQOffset + GMAX * kQRow;
    static constexpr int kSmem = kPOffset + NCW * kPBytes + 1024;  // + slack for 1 KiB alignment
    static_assert(kMergeBytes <= kBarOffset, "merge buffer must fit in the stage ring");
    static_assert(NCW % kSplit == 0 && NSTAGE % kTeams == 0, "each stage is always consumed by the same team");
    static_assert(kQOffset % 16 == 0, "16-byte loads of the staged q");
};

// One warp's online-softmax state for g <= GMAX query heads of a kv head (all of the
// group's, or one warp's share of them), over fp32 K/V tiles staged as F32Cfg lays them
// out. Scores: lane (quarter h4 = lane / 8, token t8 = lane % 8) dots its quarter of the
// head dimension for tokens t8 and t8 + 8 with every head's query (packed fp32 pairs),
// then two shuffles add the quarters. The softmax weights go through the warp's
// shared-memory slot so that P V can take four tokens' weights of a head in one
// broadcast load; lane l accumulates head-dim elements kDims l .. kDims l + kDims - 1 of
// every head.
template <int D, int GMAX>
struct WarpAttnF32 {
    static constexpr int kSubBytes = kBlock * 128;  // 2 KiB: 16 rows of 32 fp32
    static constexpr int kQC = D / 16;        // 16-byte chunks in a quarter row
    static constexpr int kDims = D / 32;      // output elements per lane (4 or 2)
    static constexpr int kQuarterBytes = D + 16;
    static constexpr int kQRow = 4 * kQuarterBytes;
    static constexpr int kHG = GMAX <= 4 ? GMAX : 4;  // heads per group
    float m[GMAX], l[GMAX];
    uint64_t acc[GMAX][kDims / 2];
    uint32_t q_s, p_s;  // shared addresses: staged query rows, this warp's weights
    int g;

    __device__ __forceinline__ void init(uint32_t q_smem, uint32_t p_smem, int group) {
        q_s = q_smem;
        p_s = p_smem;
        g = group;
    }

    __device__ __forceinline__ void reset() {
#pragma unroll
        for (int h = 0; h < GMAX; ++h) {
            m[h] = -INFINITY;
            l[h] = 0.f;
#pragma unroll
            for (int i = 0; i < kDims / 2; ++i) acc[h][i] = 0;
        }
    }

    // Rows below `lo` of the staged tiles are not tokens of the sequence (zero-filled by TMA).
    // Heads go in groups of kHG (scores, softmax, then P V per group): fewer registers at
    // the price of reading the block's K and V tiles from shared memory once per group.
    __device__ __forceinline__ void block(uint32_t sk, uint32_t sv, int lo, float scale_log2, int lane, int = 0,
                                          int = 0, bool = false) {
        const int h4 = lane >> 3, t8 = lane & 7;
        constexpr int kLaneBytes = kDims * 4;
        const int ci_v = (lane * kLaneBytes) >> 4;
        const uint32_t vbase = sv + (ci_v >> 3) * kSubBytes + ((lane * kLaneBytes) & 15);
        const int cv = ci_v & 7;
#pragma unroll
        for (int hg = 0; hg < GMAX; hg += kHG) {
            if (hg >= g) break;
            uint64_t da[kHG], db[kHG];  // partial dot products, tokens t8 and t8 + 8
#pragma unroll
            for (int k = 0; k < kHG; ++k) da[k] = db[k] = 0;
#pragma unroll
            for (int j = 0; j < kQC; ++j) {
                const int ci = h4 * kQC + j;  // 16-byte chunk of the row
                const int u = ci >> 3, c = ci & 7;
                const uint32_t at = sk + u * kSubBytes + ((c ^ t8) << 4);  // rows t8, t8 + 8 share the swizzle
                uint32_t x[4], y[4];
                ld_shared_v4(at + t8 * 128, x);
                ld_shared_v4(at + (t8 + 8) * 128, y);
                const uint64_t x01 = pack_f2(__uint_as_float(x[0]), __uint_as_float(x[1]));
                const uint64_t x23 = pack_f2(__uint_as_float(x[2]), __uint_as_float(x[3]));
                const uint64_t y01 = pack_f2(__uint_as_float(y[0]), __uint_as_float(y[1]));
                const uint64_t y23 = pack_f2(__uint_as_float(y[2]), __uint_as_float(y[3]));
#pragma unroll
                for (int k = 0; k < kHG; ++k) {
                    if (hg + k < g) {
                        uint32_t qv[4];
                        ld_shared_v4(q_s + (hg + k) * kQRow + h4 * kQuarterBytes + j * 16, qv);
                        const uint64_t q01 = pack_f2(__uint_as_float(qv[0]), __uint_as_float(qv[1]));
                        const uint64_t q23 = pack_f2(__uint_as_float(qv[2]), __uint_as_float(qv[3]));
                        da[k] = fma_f2(x23, q23, fma_f2(x01, q01, da[k]));
                        db[k] = fma_f2(y23, q23, fma_f2(y01, q01, db[k]));
                    }
                }
            }
#pragma unroll
            for (int k = 0; k < kHG; ++k) {
                const int h = hg + k;
                if (h < g) {
                    float a0, a1, b0, b1;
                    unpack_f2(da[k], a0, a1);
                    unpack_f2(db[k], b0, b1);
                    float s0 = a0 + a1, s1 = b0 + b1;
                    s0 += __shfl_xor_sync(0xffffffffu, s0, 8);
                    s1 += __shfl_xor_sync(0xffffffffu, s1, 8);
                    s0 += __shfl_xor_sync(0xffffffffu, s0, 16);
                    s1 += __shfl_xor_sync(0xffffffffu, s1, 16);
                    const float x0 = t8 >= lo ? s0 * scale_log2 : -INFINITY;
                    const float x1 = t8 + 8 >= lo ? s1 * scale_log2 : -INFINITY;
                    float mx = fmaxf(x0, x1);
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                    const float mn = fmaxf(m[h], mx);        // finite: a block holds at least one token
                    const float al = ex2_approx(m[h] - mn);  // 0 on the first block (m = -inf)
                    const float p0 = ex2_approx(x0 - mn), p1 = ex2_approx(x1 - mn);
                    m[h] = mn;
                    l[h] = l[h] * al + (h4 == 0 ? p0 + p1 : 0.f);
                    const uint64_t al2 = pack_f2(al, al);
#pragma unroll
                    for (int i = 0; i < kDims / 2; ++i) acc[h][i] = fma_f2(acc[h][i], al2, 0);
                    if (h4 == (k & 3)) {  // one quarter of the lanes writes the head's weights
                        asm volatile("st.shared.f32 [%0], %1;" ::"r"(p_s + (h * kBlock + t8) * 4), "f"(p0) : "memory");
                        asm volatile("st.shared.f32 [%0], %1;" ::"r"(p_s + (h * kBlock + t8 + 8) * 4), "f"(p1)
                                     : "memory");
                    }
                }
            }
            __syncwarp();
            // P V: this lane's kDims elements of every token's V row, the group's heads
#pragma unroll
            for (int t4 = 0; t4 < kBlock; t4 += 4) {
                float pw[kHG][4];
#pragma unroll
                for (int k = 0; k < kHG; ++k) {
                    if (hg + k < g) {
                        uint32_t w[4];
                        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                                     : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                                     : "r"(p_s + ((hg + k) * kBlock + t4) * 4)
                                     : "memory");
#pragma unroll
                        for (int e = 0; e < 4; ++e) pw[k][e] = __uint_as_float(w[e]);
                    }
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int t = t4 + e;
                    const uint32_t at = vbase + t * 128 + ((cv ^ (t & 7)) << 4);
                    uint64_t v2[kDims / 2];
                    if constexpr (kDims == 4) {
                        uint32_t w[4];
                        ld_shared_v4(at, w);
                        v2[0] = pack_f2(__uint_as_float(w[0]), __uint_as_float(w[1]));
                        v2[1] = pack_f2(__uint_as_float(w[2]), __uint_as_float(w[3]));
                    } else {
                        uint32_t w[2];
                        ld_shared_v2(at, w);
                        v2[0] = pack_f2(__uint_as_float(w[0]), __uint_as_float(w[1]));
                    }
#pragma unroll
                    for (int k = 0; k < kHG; ++k) {
                        if (hg + k < g) {
                            const uint64_t p2 = pack_f2(pw[k][e], pw[k][e]);
#pragma unroll
                            for (int i = 0; i < kDims / 2; ++i) acc[hg + k][i] = fma_f2(v2[i], p2, acc[hg + k][i]);
                        }
                    }
                }
            }
        }
        __syncwarp();  // the weights' slot is rewritten by the next block
    }

    __device__ __forceinline__ void reduce_l() {
#pragma unroll
        for (int h = 0; h < GMAX; ++h)
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) l[h] += __shfl_xor_sync(0xffffffffu, l[h], o);
    }

    // Rows h < GMAX of the merge buffer (rows past the warp's heads are never read).
    __device__ __forceinline__ void store_merge(float *ml, float *acc_rows, int stride, int lane) const {
#pragma unroll
        for (int h = 0; h < GMAX; ++h) {
            if (lane == 0) {
                ml[h * 2 + 0] = m[h];
                ml[h * 2 + 1] = l[h];
            }
#pragma unroll
            for (int i = 0; i < kDims / 2; ++i) {
                float a, b;
                unpack_f2(acc[h][i], a, b);
                acc_rows[h * stride + kDims * lane + 2 * i] = a;
                acc_rows[h * stride + kDims * lane + 2 * i + 1] = b;
            }
        }
    }
};

// From a query-head bound of PKV_F32_SPLIT_FROM on, each block is split between the two
// warps of a team (each takes half the heads on the same staged tiles): a block's
// CUDA-core work is halved, and each team alternates between two stages, so a warp's
// next block is in flight while it computes.
template <int D, int GMAX, int NSTAGE, int NCW>
__global__ void __launch_bounds__((NCW + 1) * 32, GMAX >= 16 ? 1 : (GMAX >= 8 ? 2 : 3))
    decode_f32_staged_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                             const DecodeParams p) {
    using C = F32Cfg<D, GMAX, NSTAGE, NCW>;
    constexpr int GW = C::kWarpHeads;
    extern __shared__ uint8_t smem_raw[];

    const int part = blockIdx.x, h = blockIdx.y, s = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = p.group;
    const int len = seq_len(p, s, tid == 0 && part == 0 && h == 0);
    const int nblk = (len + kBlock - 1) / kBlock;
    const int npart = (nblk + p.part_blocks - 1) / p.part_blocks;
    float *out = static_cast<float *>(p.out);

    if (len == 0) {  // empty context: zero output rows
        if (part == 0) {
            float *o = out + ((size_t)s * p.num_q_heads + (size_t)h * g) * D;
            for (int i = tid; i < g * D; i += C::kThreads) o[i] = 0.f;
        }
        return;
    }
    if (part >= npart) return;

    const int b_begin = part * p.part_blocks;
    const int nb = min(nblk - b_begin, p.part_blocks);
    const int last_valid = len - (nblk - 1) * kBlock;  // tokens in the sequence's last block

    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(base + C::kBarOffset);
    uint64_t *empty = full + NSTAGE;
    if (tid == 0) {
        prefetch_tensormap(&tmk);
        prefetch_tensormap(&tmv);
        for (int i = 0; i < NSTAGE; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], C::kSplit);
        }
        mbar_fence_init();
    }
    // the group's query rows: quarter r of head row hh at q_smem + hh kQRow + r kQuarterBytes
    const float *qg = static_cast<const float *>(p.q) + ((size_t)s * p.num_q_heads + (size_t)h * g) * D;
    for (int i = tid; i < g * (D / 4); i += C::kThreads) {  // 16-byte pieces
        const int hh = i / (D / 4), k = i - hh * (D / 4);  // piece k of row hh: quarter k / (D / 16)
        const float4 v = __ldg(reinterpret_cast<const float4 *>(qg + (size_t)hh * D) + k);
        *reinterpret_cast<float4 *>(base + C::kQOffset + hh * C::kQRow + (k / (D / 16)) * C::kQuarterBytes +
                                    (k % (D / 16)) * 16) = v;
    }
    __syncthreads();

    if (warp == NCW) {
        grid_produce<C, NSTAGE>(tmk, tmv, p.block_tables + (size_t)s * p.max_blocks_per_seq, b_begin, nb, nblk - 1,
                                last_valid, p.num_blocks, p.num_kv_heads, h, base, full, empty, lane);
        return;
    }
    // team `team` takes blocks team, team + kTeams, ...; its member `mem` the heads
    // mem GW .. mem GW + GW - 1 of the group
    const int team = warp / C::kSplit, mem = warp % C::kSplit;
    const int h0 = mem * GW;
    const int nh = min(GW, g - h0);
    WarpAttnF32<D, GW> wa;
    wa.init(smem_u32(base + C::kQOffset + h0 * C::kQRow), smem_u32(base + C::kPOffset + warp * C::kPBytes), nh);
    wa.reset();
    const int last_in_range = (b_begin + nb - 1 == nblk - 1) ? nb - 1 : -1;
    for (int j = team; j < nb; j += C::kTeams) {
        const int st = j % NSTAGE;
        if (!mbar_wait(&full[st], (j / NSTAGE) & 1)) {
            raise_error(PKV_DEVERR_TIMEOUT);
            break;
        }
        const uint32_t sk = smem_u32(base + st * C::kStage);
        wa.block(sk, sk + C::kTile, j == last_in_range ? kBlock - last_valid : 0, p.scale_log2, lane);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
    }
    wa.reduce_l();
    named_barrier_sync(1, NCW * 32);  // every consumer is done with the stage ring
    float *mml = reinterpret_cast<float *>(base);   // [NCW][GW][2]
    float *macc = mml + NCW * GW * 2;                // [NCW][GW][kMergeStride]
    wa.store_merge(mml + warp * GW * 2, macc + warp * GW * C::kMergeStride, C::kMergeStride, lane);
    named_barrier_sync(1, NCW * 32);
    const size_t orow0 = (size_t)s * p.num_q_heads + (size_t)h * g;
    for (int idx = tid; idx < g * D; idx += NCW * 32) {
        const int col = idx / D, d = idx - col * D;
        const int cm = col / GW, k = col - cm * GW;  // the member holding the column, its row there
        float M = -INFINITY;
#pragma unroll
        for (int t = 0; t < C::kTeams; ++t) M = fmaxf(M, mml[((t * C::kSplit + cm) * GW + k) * 2]);
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int t = 0; t < C::kTeams; ++t) {
            const int r = (t * C::kSplit + cm) * GW + k;
            const float mw = mml[r * 2];
            const float f = (mw == -INFINITY) ? 0.f : ex2_approx(mw - M);
            L += mml[r * 2 + 1] * f;
            O += macc[r * C::kMergeStride + d] * f;
        }
        const float o = O / L;
        if (npart == 1) {
            out[(orow0 + col) * D + d] = o;
        } else {
            const size_t r = (orow0 + col) * p.max_parts + part;
            p.ws_o[r * D + d] = o;
            if (d == 0) {
                p.ws_ml[r * 2 + 0] = M;
                p.ws_ml[r * 2 + 1] = L;
            }
        }
    }
}

// =====================================================================================
// K1 (fp32, staged, tensor cores): the staged kernel's decomposition for groups of 5..16
// query heads, with the per-block products on the tensor cores in tf32 split three ways.
// An fp32 value x is hi + lo: hi = x rounded to tf32 (a 10-bit significand), lo = x - hi
// exactly; the tensor core keeps lo to tf32 as well, so lo's dropped bits are below 2^-21
// of x. A product a b is taken as ah bh + ah bl + al bh (three m16n8k8 MMAs with fp32
// accumulation); the dropped al bl is below 2^-20 of |a b|.
// =====================================================================================
__device__ __forceinline__ void tf32_split(float x, uint32_t &hi, uint32_t &lo) {
    uint32_t h;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(h) : "f"(x));
    hi = h;
    lo = __float_as_uint(x - __uint_as_float(h));
}

// D = A(16x8, row) * B(8x8, col) + D, tf32 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_tf32_1688(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// d += a b with a and b split as above
__device__ __forceinline__ void mma_tf32x3(float (&d)[4], const uint32_t (&ah)[4], const uint32_t (&al)[4],
                                           uint32_t bh0, uint32_t bh1, uint32_t bl0, uint32_t bl1) {
    mma_tf32_1688(d, al, bh0, bh1);
    mma_tf32_1688(d, ah, bl0, bl1);
    mma_tf32_1688(d, ah, bh0, bh1);
}

// One warp's online-softmax state for the GMAX (8 or 16) query-head columns of a kv head
// (columns past the group are zero queries, never read back), over fp32 K/V tiles staged as
// F32Cfg lays them out. Per block: S^T (16 tokens x 8 heads per n-tile) = K Q^T, K
// fragments by ldmatrix from the swizzled tile (a 32-bit element is a pair of b16), Q^T
// fragments split once per CTA into shared memory; the softmax on the S^T fragments;
// the weights through the warp's shared-memory slot into P^T fragments; then
// O^T (D x 8 per n-tile) += V^T P^T with V^T fragments read element by element.
template <int D, int GMAX>
struct WarpAttnTF32 {
    static constexpr int kNT = GMAX / 8;          // n-tiles of 8 query heads
    static constexpr int kKS = D / 8;             // k-steps of S^T = K Q^T
    static constexpr int kMT = D / 16;            // m-tiles of O^T
    static constexpr int kSubBytes = kBlock * 128;
    static constexpr int kHeadStride = 20;        // floats per head row of the weight slot (banks spread)
    static constexpr int kQBytes = kNT * kKS * 32 * 16;          // split Q^T fragments, per lane 16 bytes
    static constexpr int kPBytes = kNT * 8 * kHeadStride * 4;    // one warp's weights of a block
    float m[kNT][2], l[kNT][2];   // columns nt 8 + 2 t and + 1 (t = lane % 4); l over this lane's tokens
    float acc[kNT][kMT][4];       // O^T fragments: rows (dims) 16 mi + lane / 4 (+ 8), columns 2 t (+ 1)
    uint32_t q_s, p_s;

    // All threads of the CTA: the group's q (g heads at qg, D floats each) as split B
    // fragments of S^T = K Q^T: entry (nt, ks, lane) holds hi and lo of q[head][8 ks + t]
    // and q[head][8 ks + t + 4], head = 8 nt + lane / 4, t = lane % 4 (zero past the group).
    static __device__ __forceinline__ void stage_q(uint8_t *dst, const float *qg, int g, int tid, int nthreads) {
        for (int i = tid; i < kNT * kKS * 32; i += nthreads) {
            const int ln = i & 31, ks = (i >> 5) % kKS, nt = i / (32 * kKS);
            const int head = nt * 8 + (ln >> 2), dim = 8 * ks + (ln & 3);
            const float b0 = head < g ? __ldg(qg + (size_t)head * D + dim) : 0.f;
            const float b1 = head < g ? __ldg(qg + (size_t)head * D + dim + 4) : 0.f;
            uint32_t h0, l0, h1, l1;
            tf32_split(b0, h0, l0);
            tf32_split(b1, h1, l1);
            *reinterpret_cast<uint4 *>(dst + (size_t)i * 16) = make_uint4(h0, h1, l0, l1);
        }
    }

    __device__ __forceinline__ void init(uint32_t q_smem, uint32_t p_smem) {
        q_s = q_smem;
        p_s = p_smem;
    }

    __device__ __forceinline__ void reset() {
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt) {
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                m[nt][hh] = -INFINITY;
                l[nt][hh] = 0.f;
            }
#pragma unroll
            for (int mi = 0; mi < kMT; ++mi)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[nt][mi][e] = 0.f;
        }
    }

    // Rows below `lo` of the staged tiles are not tokens of the sequence (zero-filled by TMA).
    __device__ __forceinline__ void block(uint32_t sk, uint32_t sv, int lo, float scale_log2, int lane) {
        const int gq = lane >> 2, t = lane & 3;
        // S^T = K Q^T
        float sacc[kNT][4];
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) sacc[nt][e] = 0.f;
        // ldmatrix rows: lanes 8 m .. 8 m + 7 address matrix m = (token rows 8 (m & 1) .., 16-byte
        // chunk m >> 1 of the k-step's two)
        const int mrow = ((lane >> 3) & 1) * 8 + (lane & 7), mhalf = lane >> 4;
#pragma unroll
        for (int ks = 0; ks < kKS; ++ks) {
            const int ch = 2 * (ks & 3) + mhalf;
            uint32_t a[4], ah[4], al[4];
            ldsm_x4(sk + (ks >> 2) * kSubBytes + mrow * 128 + ((ch ^ (mrow & 7)) << 4), a);
#pragma unroll
            for (int i = 0; i < 4; ++i) tf32_split(__uint_as_float(a[i]), ah[i], al[i]);
#pragma unroll
            for (int nt = 0; nt < kNT; ++nt) {
                uint32_t qb[4];
                ld_shared_v4(q_s + ((nt * kKS + ks) * 32 + lane) * 16, qb);
                mma_tf32x3(sacc[nt], ah, al, qb[0], qb[1], qb[2], qb[3]);
            }
        }
        // online softmax per column; lane holds tokens gq, gq + 8 of columns 2 t, 2 t + 1
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt) {
            const float x00 = gq >= lo ? sacc[nt][0] * scale_log2 : -INFINITY;
            const float x01 = gq >= lo ? sacc[nt][1] * scale_log2 : -INFINITY;
            const float x10 = gq + 8 >= lo ? sacc[nt][2] * scale_log2 : -INFINITY;
            const float x11 = gq + 8 >= lo ? sacc[nt][3] * scale_log2 : -INFINITY;
            float mx0 = fmaxf(x00, x10), mx1 = fmaxf(x01, x11);
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
            }
            const float mn0 = fmaxf(m[nt][0], mx0), mn1 = fmaxf(m[nt][1], mx1);  // finite: a block has a token
            const float al0 = ex2_approx(m[nt][0] - mn0), al1 = ex2_approx(m[nt][1] - mn1);
            m[nt][0] = mn0;
            m[nt][1] = mn1;
            const float p00 = ex2_approx(x00 - mn0), p10 = ex2_approx(x10 - mn0);
            const float p01 = ex2_approx(x01 - mn1), p11 = ex2_approx(x11 - mn1);
            l[nt][0] = l[nt][0] * al0 + (p00 + p10);
            l[nt][1] = l[nt][1] * al1 + (p01 + p11);
#pragma unroll
            for (int mi = 0; mi < kMT; ++mi) {
                acc[nt][mi][0] *= al0;
                acc[nt][mi][2] *= al0;
                acc[nt][mi][1] *= al1;
                acc[nt][mi][3] *= al1;
            }
            // weights into the slot as [column][token]
            const uint32_t ps = p_s + nt * 8 * kHeadStride * 4;
            asm volatile("st.shared.f32 [%0], %1;" ::"r"(ps + ((2 * t) * kHeadStride + gq) * 4), "f"(p00) : "memory");
            asm volatile("st.shared.f32 [%0], %1;" ::"r"(ps + ((2 * t + 1) * kHeadStride + gq) * 4), "f"(p01)
                         : "memory");
            asm volatile("st.shared.f32 [%0], %1;" ::"r"(ps + ((2 * t) * kHeadStride + gq + 8) * 4), "f"(p10)
                         : "memory");
            asm volatile("st.shared.f32 [%0], %1;" ::"r"(ps + ((2 * t + 1) * kHeadStride + gq + 8) * 4), "f"(p11)
                         : "memory");
        }
        __syncwarp();
        // O^T += V^T P^T, 8 tokens per k-step
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
            uint32_t bh[kNT][2], bl[kNT][2];  // P^T fragments: tokens 8 kk + t (+ 4), column gq
#pragma unroll
            for (int nt = 0; nt < kNT; ++nt) {
                const uint32_t ps = p_s + nt * 8 * kHeadStride * 4 + (gq * kHeadStride + 8 * kk + t) * 4;
                float w0, w1;
                asm volatile("ld.shared.f32 %0, [%1];" : "=f"(w0) : "r"(ps) : "memory");
                asm volatile("ld.shared.f32 %0, [%1];" : "=f"(w1) : "r"(ps + 16) : "memory");
                tf32_split(w0, bh[nt][0], bl[nt][0]);
                tf32_split(w1, bh[nt][1], bl[nt][1]);
            }
            const int t0 = 8 * kk + t, t1 = t0 + 4;
#pragma unroll
            for (int mi = 0; mi < kMT; ++mi) {
                // V^T fragment: rows (dims) 16 mi + gq (+ 8), columns (tokens) t0, t1
                const int d0 = 16 * mi + gq, d1 = d0 + 8;
                const uint32_t a0 = sv + (d0 >> 5) * kSubBytes + t0 * 128 + ((((d0 & 31) >> 2) ^ (t0 & 7)) << 4) + (d0 & 3) * 4;
                const uint32_t a1 = sv + (d1 >> 5) * kSubBytes + t0 * 128 + ((((d1 & 31) >> 2) ^ (t0 & 7)) << 4) + (d1 & 3) * 4;
                const uint32_t a2 = sv + (d0 >> 5) * kSubBytes + t1 * 128 + ((((d0 & 31) >> 2) ^ (t1 & 7)) << 4) + (d0 & 3) * 4;
                const uint32_t a3 = sv + (d1 >> 5) * kSubBytes + t1 * 128 + ((((d1 & 31) >> 2) ^ (t1 & 7)) << 4) + (d1 & 3) * 4;
                float v[4];
                asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v[0]) : "r"(a0));
                asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v[1]) : "r"(a1));
                asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v[2]) : "r"(a2));
                asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v[3]) : "r"(a3));
                uint32_t ah[4], al[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) tf32_split(v[i], ah[i], al[i]);
#pragma unroll
                for (int nt = 0; nt < kNT; ++nt)
                    mma_tf32x3(acc[nt][mi], ah, al, bh[nt][0], bh[nt][1], bl[nt][0], bl[nt][1]);
            }
        }
        __syncwarp();  // the weights' slot is rewritten by the next block
    }

    __device__ __forceinline__ void reduce_l() {
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                for (int o = 4; o < 32; o <<= 1) l[nt][hh] += __shfl_xor_sync(0xffffffffu, l[nt][hh], o);
    }

    // Rows (columns of the group) 0 .. GMAX - 1 of the merge buffer.
    __device__ __forceinline__ void store_merge(float *ml, float *acc_rows, int stride, int lane) const {
        const int gq = lane >> 2, t = lane & 3;
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int col = nt * 8 + 2 * t + hh;
                if (gq == 0) {
                    ml[col * 2 + 0] = m[nt][hh];
                    ml[col * 2 + 1] = l[nt][hh];
                }
#pragma unroll
                for (int mi = 0; mi < kMT; ++mi) {
                    acc_rows[col * stride + 16 * mi + gq] = acc[nt][mi][hh];
                    acc_rows[col * stride + 16 * mi + gq + 8] = acc[nt][mi][2 + hh];
                }
            }
    }
};

template <int D, int GMAX, int NSTAGE, int NCW>
struct F32TcCfg {
    using WA = WarpAttnTF32<D, GMAX>;
    static constexpr int kTile = kBlock * D * 4;
    static constexpr int kStage = 2 * kTile;
    static constexpr int kThreads = (NCW + 1) * 32;
    static constexpr int kMergeStride = D + 4;
    static constexpr int kMergeBytes = NCW * GMAX * (2 + kMergeStride) * 4;
    static constexpr int kBarOffset = NSTAGE * kStage;
    static constexpr int kQOffset = kBarOffset + 2 * NSTAGE * 8;
    static constexpr int kPOffset = kQOffset + WA::kQBytes;
    static constexpr int kSmem = kPOffset + NCW * WA::kPBytes + 1024;  // + slack for 1 KiB alignment
    static_assert(kMergeBytes <= kBarOffset, "merge buffer must fit in the stage ring");
    static_assert(NSTAGE % NCW == 0, "each stage is always consumed by the same warp");
    static_assert(kQOffset % 16 == 0 && WA::kPBytes % 16 == 0, "16-byte aligned areas");
};

template <int D, int GMAX, int NSTAGE, int NCW>
__global__ void __launch_bounds__((NCW + 1) * 32)
    decode_f32_tc_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                         const DecodeParams p) {
    using C = F32TcCfg<D, GMAX, NSTAGE, NCW>;
    extern __shared__ uint8_t smem_raw[];

    const int part = blockIdx.x, h = blockIdx.y, s = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = p.group;
    const int len = seq_len(p, s, tid == 0 && part == 0 && h == 0);
    const int nblk = (len + kBlock - 1) / kBlock;
    const int npart = (nblk + p.part_blocks - 1) / p.part_blocks;
    float *out = static_cast<float *>(p.out);

    if (len == 0) {  // empty context: zero output rows
        if (part == 0) {
            float *o = out + ((size_t)s * p.num_q_heads + (size_t)h * g) * D;
            for (int i = tid; i < g * D; i += C::kThreads) o[i] = 0.f;
        }
        return;
    }
    if (part >= npart) return;

    const int b_begin = part * p.part_blocks;
    const int nb = min(nblk - b_begin, p.part_blocks);
    const int last_valid = len - (nblk - 1) * kBlock;  // tokens in the sequence's last block

    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(base + C::kBarOffset);
    uint64_t *empty = full + NSTAGE;
    if (tid == 0) {
        prefetch_tensormap(&tmk);
        prefetch_tensormap(&tmv);
        for (int i = 0; i < NSTAGE; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        mbar_fence_init();
    }
    const float *qg = static_cast<const float *>(p.q) + ((size_t)s * p.num_q_heads + (size_t)h * g) * D;
    C::WA::stage_q(base + C::kQOffset, qg, g, tid, C::kThreads);
    __syncthreads();

    if (warp == NCW) {
        grid_produce<C, NSTAGE>(tmk, tmv, p.block_tables + (size_t)s * p.max_blocks_per_seq, b_begin, nb, nblk - 1,
                                last_valid, p.num_blocks, p.num_kv_heads, h, base, full, empty, lane);
        return;
    }
    typename C::WA wa;
    wa.init(smem_u32(base + C::kQOffset), smem_u32(base + C::kPOffset + warp * C::WA::kPBytes));
    wa.reset();
    const int last_in_range = (b_begin + nb - 1 == nblk - 1) ? nb - 1 : -1;
    for (int j = warp; j < nb; j += NCW) {
        const int st = j % NSTAGE;
        if (!mbar_wait(&full[st], (j / NSTAGE) & 1)) {
            raise_error(PKV_DEVERR_TIMEOUT);
            break;
        }
        const uint32_t sk = smem_u32(base + st * C::kStage);
        wa.block(sk, sk + C::kTile, j == last_in_range ? kBlock - last_valid : 0, p.scale_log2, lane);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
    }
    wa.reduce_l();
    named_barrier_sync(1, NCW * 32);  // every consumer is done with the stage ring
    float *mml = reinterpret_cast<float *>(base);   // [NCW][GMAX][2]
    float *macc = mml + NCW * GMAX * 2;              // [NCW][GMAX][kMergeStride]
    wa.store_merge(mml + warp * GMAX * 2, macc + warp * GMAX * C::kMergeStride, C::kMergeStride, lane);
    named_barrier_sync(1, NCW * 32);
    const size_t orow0 = (size_t)s * p.num_q_heads + (size_t)h * g;
    for (int idx = tid; idx < g * D; idx += NCW * 32) {
        const int col = idx / D, d = idx - col * D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NCW; ++w) M = fmaxf(M, mml[(w * GMAX + col) * 2]);
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < NCW; ++w) {
            const float mw = mml[(w * GMAX + col) * 2];
            const float f = (mw == -INFINITY) ? 0.f : ex2_approx(mw - M);
            L += mml[(w * GMAX + col) * 2 + 1] * f;
            O += macc[(w * GMAX + col) * C::kMergeStride + d] * f;
        }
        const float o = O / L;
        if (npart == 1) {
            out[(orow0 + col) * D + d] = o;
        } else {
            const size_t r = (orow0 + col) * p.max_parts + part;
            p.ws_o[r * D + d] = o;
            if (d == 0) {
                p.ws_ml[r * 2 + 0] = M;
                p.ws_ml[r * 2 + 1] = L;
            }
        }
    }
}

// =====================================================================================
// K2: log-sum-exp merge of a sequence's partitions, one CTA of D threads per
// (query head, sequence):  M = max_p m_p;  w_p = l_p 2^(m_p - M);
//   out = sum_p w_p o_p / sum_p w_p.
// Sequences with a single partition were written by K1 and are skipped.
// =====================================================================================

template <typename OutT, int D, int PG>
__global__ void __launch_bounds__(D *PG) lse_reduce_kernel(const DecodeParams p) {
    // PG groups of D threads: group k sums partitions k, k + PG, ...
    extern __shared__ float rsm[];  // [32] scratch, [PG][D] group sums, [max_parts] weights
    const int hq = blockIdx.x, s = blockIdx.y, tid = threadIdx.x;
    const int d = tid % D, grp = tid / D;
    const int len = seq_len(p, s, false);
    const int nblk = (len + kBlock - 1) / kBlock;
    const int npart = (nblk + p.part_blocks - 1) / p.part_blocks;
    if (npart <= 1) return;
    const size_t row = (size_t)s * p.num_q_heads + hq;
    const float *ml = p.ws_ml + row * p.max_parts * 2;
    const float *o = p.ws_o + row * p.max_parts * D;
    float *scratch = rsm;
    float *gsum = rsm + 32;
    float *w = gsum + PG * D;
    float M = -INFINITY;
    for (int i = tid; i < npart; i += D * PG) M = fmaxf(M, ml[2 * i]);
    M = block_reduce(M, true, scratch);
    float W = 0.f;
    for (int i = tid; i < npart; i += D * PG) {
        const float wi = ml[2 * i + 1] * exp2f(ml[2 * i] - M);
        w[i] = wi;
        W += wi;
    }
    W = block_reduce(W, false, scratch);
    __syncthreads();
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
    int i = grp;
    for (; i + 3 * PG < npart; i += 4 * PG) {
        a0 = fmaf(w[i], o[(size_t)i * D + d], a0);
        a1 = fmaf(w[i + PG], o[(size_t)(i + PG) * D + d], a1);
        a2 = fmaf(w[i + 2 * PG], o[(size_t)(i + 2 * PG) * D + d], a2);
        a3 = fmaf(w[i + 3 * PG], o[(size_t)(i + 3 * PG) * D + d], a3);
    }
    for (; i < npart; i += PG) a0 = fmaf(w[i], o[(size_t)i * D + d], a0);
    gsum[grp * D + d] = (a0 + a1) + (a2 + a3);
    __syncthreads();
    if (grp == 0) {
        float r = 0.f;
#pragma unroll
        for (int k = 0; k < PG; ++k) r += gsum[k * D + d];
        r /= W;
        OutT *out = static_cast<OutT *>(p.out);
        if constexpr (sizeof(OutT) == 2) {
            out[row * D + d] = __float2bfloat16_rn(r);
        } else {
            out[row * D + d] = r;
        }
    }
}

// =====================================================================================
// K3: KV append. One thread per 16-byte vector of (token, kv head, head-dim
// chunk), so even a one-token-per-sequence step spreads over many CTAs.
// =====================================================================================
__global__ void kv_append_kernel(const uint4 *__restrict__ k, const uint4 *__restrict__ v,
                                 const int64_t *__restrict__ slots, uint4 *__restrict__ kc, uint4 *__restrict__ vc,
                                 int num_tokens, int num_kv_heads, int vec_per_row, int num_blocks) {
    pdl_trigger();  // a decode step's attention kernel may start its set-up now; it waits for the writes
    const int per_token = num_kv_heads * vec_per_row;
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (long long)num_tokens * per_token) return;
    const int t = (int)(idx / per_token);
    const int rem = (int)(idx - (long long)t * per_token);
    const int64_t slot = __ldg(slots + t);
    if (slot < 0) return;
    if (slot >= (int64_t)num_blocks * kBlock) {
        if (rem == 0) raise_error(PKV_DEVERR_SLOT);
        return;
    }
    const int hh = rem / vec_per_row, c = rem - hh * vec_per_row;
    const size_t dst = ((((size_t)(slot >> 4)) * num_kv_heads + hh) * kBlock + (slot & 15)) * vec_per_row + c;
    kc[dst] = __ldg(k + idx);
    vc[dst] = __ldg(v + idx);
}

// =====================================================================================
// K4: whole-block moves. For each (src, dst) pair, block src of a source pool
// is copied onto block dst of a destination pool -- every kv head, all 16
// slots -- for each of `ncache` caches (K and V of one or more layers). The
// pools are the same for copy-on-write, different for swapping to and from a
// host pool (pinned host memory the GPU addresses directly) or between device
// pools. grid (chunks, pairs, caches); 16-byte vectors.
// =====================================================================================
struct BlockMove {
    const uint4 *src[2];                // K and V of one layer, given inline ...
    uint4 *dst[2];
    const uint4 *const *src_k_layers;   // ... or per-layer pointer arrays [layers]
    const uint4 *const *src_v_layers;
    uint4 *const *dst_k_layers;
    uint4 *const *dst_v_layers;
    int src_num_blocks, dst_num_blocks;
    int64_t vec_per_block;
};

__global__ void move_blocks_kernel(const BlockMove m, const int64_t *__restrict__ pairs) {
    const int pr = blockIdx.y, c = blockIdx.z;
    const int64_t src = __ldg(pairs + 2 * pr), dst = __ldg(pairs + 2 * pr + 1);
    const bool lead = threadIdx.x == 0 && blockIdx.x == 0;
    if (src < 0 || src >= m.src_num_blocks || dst < 0 || dst >= m.dst_num_blocks) {
        if (lead && c == 0) raise_error(PKV_DEVERR_PAIR);
        return;
    }
    const uint4 *sb;
    uint4 *db;
    if (m.src_k_layers) {
        const int layer = c >> 1;
        sb = (c & 1) ? m.src_v_layers[layer] : m.src_k_layers[layer];
        db = (c & 1) ? m.dst_v_layers[layer] : m.dst_k_layers[layer];
        if (((reinterpret_cast<uintptr_t>(sb) | reinterpret_cast<uintptr_t>(db)) & 15) != 0 || !sb || !db) {
            if (lead && pr == 0) raise_error(PKV_DEVERR_POINTER);
            return;
        }
    } else {
        sb = m.src[c];
        db = m.dst[c];
    }
    const uint4 *sp = sb + src * m.vec_per_block;
    uint4 *dp = db + dst * m.vec_per_block;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < m.vec_per_block;
         i += (int64_t)gridDim.x * blockDim.x)
        dp[i] = sp[i];
}

// K3 for several layers at once: grid (vector chunks, layers); layer l reads
// k[l], v[l] ([T][Hkv][D]) and writes k_caches[l], v_caches[l] at the same slots.
__global__ void kv_append_layers_kernel(const uint4 *const *k, const uint4 *const *v, const int64_t *__restrict__ slots,
                                        uint4 *const *kc, uint4 *const *vc, int num_tokens, int num_kv_heads,
                                        int vec_per_row, int num_blocks) {
    const int layer = blockIdx.y;
    const uint4 *kl = k[layer], *vl = v[layer];
    uint4 *kcl = kc[layer], *vcl = vc[layer];
    const bool lead = threadIdx.x == 0 && blockIdx.x == 0;
    if (((reinterpret_cast<uintptr_t>(kl) | reinterpret_cast<uintptr_t>(vl) | reinterpret_cast<uintptr_t>(kcl) |
          reinterpret_cast<uintptr_t>(vcl)) & 15) != 0 || !kl || !vl || !kcl || !vcl) {
        if (lead) raise_error(PKV_DEVERR_POINTER);
        return;
    }
    const int per_token = num_kv_heads * vec_per_row;
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (long long)num_tokens * per_token) return;
    const int t = (int)(idx / per_token);
    const int rem = (int)(idx - (long long)t * per_token);
    const int64_t slot = __ldg(slots + t);
    if (slot < 0) return;
    if (slot >= (int64_t)num_blocks * kBlock) {
        if (rem == 0 && layer == 0) raise_error(PKV_DEVERR_SLOT);
        return;
    }
    const int hh = rem / vec_per_row, cc = rem - hh * vec_per_row;
    const size_t dst = ((((size_t)(slot >> 4)) * num_kv_heads + hh) * kBlock + (slot & 15)) * vec_per_row + cc;
    kcl[dst] = kl[idx];
    vcl[dst] = vl[idx];
}

// =====================================================================================
// K5: metadata checks (debug). They OR PKV_DEVERR_* bits into *err, never trap.
// =====================================================================================
__global__ void validate_tables_kernel(const int32_t *block_tables, const int32_t *context_lens, int max_blocks_per_seq,
                                       int num_blocks, int max_context_len, int32_t *err) {
    const int s = blockIdx.x;
    int len = context_lens[s];
    unsigned bits = 0;
    if (len < 0 || len > max_blocks_per_seq * kBlock || len > max_context_len) bits |= PKV_DEVERR_LENGTH;
    len = max(0, min(len, max_blocks_per_seq * kBlock));
    const int nblk = (len + kBlock - 1) / kBlock;
    for (int j = threadIdx.x; j < nblk; j += blockDim.x) {
        const int b = block_tables[(size_t)s * max_blocks_per_seq + j];
        if (b < 0 || b >= num_blocks) bits |= PKV_DEVERR_BLOCK_ID;
    }
    if (bits) atomicOr(reinterpret_cast<unsigned *>(err), bits);
}

__global__ void validate_slots_kernel(const int64_t *slots, int num_tokens, int num_blocks, int32_t *err) {
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t < num_tokens && slots[t] >= (int64_t)num_blocks * kBlock)
        atomicOr(reinterpret_cast<unsigned *>(err), PKV_DEVERR_SLOT);
}

}  // namespace pkv
