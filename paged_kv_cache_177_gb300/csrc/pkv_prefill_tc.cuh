// pkv_prefill_tc.cuh -- causal prefill attention on the 5th-generation tensor
// cores (tcgen05, accumulators and softmax weights in tensor memory).
//
// Computes what paged_prefill_attention defines ("Batching Continuo y
// PagedAttention", cruxr.ai, section "Juntándolo todo: Arquitectura de vLLM":
// the prefill pass attends each prompt token causally over the prompt, whose
// K/V sit in the paged cache): for sequence s with n new tokens, query i at
// position pos = len - n + i attends positions 0 .. pos.
//
// One CTA per (two consecutive 128-row query tiles, kv head, sequence); a
// row is a (new token, query head of the kv head's group) pair, so a tile
// holds 128 / g tokens. Keys are taken 128 at a time (8 cache blocks, a
// "chunk"), and both tiles use each staged chunk:
//
//   warp 0, one thread   TMA: both Q tiles once; per chunk its 8 K blocks and
//                        8 V blocks into two-stage rings (blocks past the
//                        sequence read as zeros; its last block is loaded from
//                        slot valid - 16 so its rows past the end are zeros)
//   warp 1, one thread   MMA, per tile t: S_t = Q_t K_j^T (128 x 128 fp32 in
//                        tensor memory), and once the softmax has turned S_t
//                        into P_t (bf16, in the same tensor-memory columns),
//                        O_t += P_t V_j with P_t read from tensor memory; the
//                        next S_t follows right after. While one tile's
//                        softmax runs, the tensor cores work on the other.
//   warps 2-3            idle (they complete warpgroup 0, which hands its
//                        registers to the softmax warpgroups)
//   warps 4-7, 8-11      softmax of tile 0 / tile 1, one thread per query row
//                        (tensor-memory lane = row): the row max of S_t, a
//                        rescale of its row of O_t when the max moved, then
//                        P_t = 2^(S_t - max) written over S_t. At the end
//                        O_t / l goes out as bf16.
//
// Tensor-core MMAs of one CTA run in issue order, so the commit that
// signals S_t of chunk j also covers P_t V of chunk j - 1: once a softmax
// thread sees S_t, its row of O_t and its P_t columns are free.
//
// The running max is lazy: the reference max of a row moves only when the
// row max exceeds it by more than 8 (in log2 units), so O is rescaled rarely
// and the weights 2^(x - reference) stay below 2^8. Softmax is invariant to
// the reference, so the result is the same.
//
// The weights of the first chunk also enter P V as their bf16 rounding
// remainder (a second P V product), as the mma.sync kernels do for positions
// < 64: rows that see only a few keys would otherwise carry the full bf16
// rounding of their weights. (Limiting it to tiles that hold such rows was
// measured slower: the extra first-chunk work staggers the two tiles'
// softmax phases, which then overlap the other tile's MMAs better.)
//
// prefill_tc_units_kernel runs the same roles with one CTA per (sequence, kv
// head) looping over all its pairs: for batches of whole prompts with many such
// units, where each pair is short and a CTA's set-up would otherwise be paid
// once per pair. It gives the remainder only in tiles holding rows that see at
// most kPrefillSplitPositions keys (the rows the remainder is for; on every tile it
// cost about 13% of the kernel's time on whole prompts: a second P V and the
// remainders' softmax work on each first chunk), its first chunk's softmax compiled
// apart from the others'. The one-pair kernel keeps the remainder on every tile's first chunk:
// there the same restriction compiled into slower code.
//
// Every wait is bounded; on a timeout the CTA records PKV_DEVERR_TIMEOUT,
// waits (bounded) for its in-flight copies and MMAs, frees its tensor memory
// and exits.
#pragma once

#include "pkv_kernels.cuh"

namespace pkv {

template <int D>
struct TcCfg {
    static constexpr int kRows = 128;                      // MMA M: query rows per tile
    static constexpr int kTiles = 2;                       // query tiles per CTA
    static constexpr int kKeys = 128;                      // MMA N of S: keys per chunk
    static constexpr int kChunkBlocks = kKeys / kBlock;    // 8
    static constexpr int kHalves = D / 64;                 // 128-byte row segments of a head vector
    static constexpr int kHalfRows = 128 * 128;            // bytes of one 128-row, 128-byte-wide region
    static constexpr int kQBytes = kRows * D * 2;          // one tile
    static constexpr int kStage = kKeys * D * 2;           // one chunk of K (or of V)
    static constexpr int kBlockBytes = kBlock * D * 2;     // one cache block of one head
    static constexpr int kStages = 2;
    static constexpr int kQOff = 0;
    static constexpr int kKOff = kQOff + kTiles * kQBytes;
    static constexpr int kVOff = kKOff + kStages * kStage;
    static constexpr int kBarOff = kVOff + kStages * kStage;
    static constexpr int kSmem = kBarOff + 256 + 1024;     // + barriers, + 1024-byte alignment slack
    static constexpr int kSoftmaxWarps = 4 * kTiles;
    static constexpr int kThreads = (4 + kSoftmaxWarps) * 32;  // warpgroup 0: TMA, MMA, 2 idle warps
    // register split (setmaxnreg): launched at kLaunchRegs each, warpgroup 0 gives
    // registers to the softmax warpgroups
    static constexpr int kLaunchRegs = 168;
    static constexpr int kLowRegs = 72;
    static constexpr int kHighRegs = 208;
    static_assert(128 * kLowRegs + kTiles * 128 * kHighRegs <= kThreads * kLaunchRegs, "register split");
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kTileCols = 256;             // per tile: S / P at +0, O at +128
    static constexpr uint32_t kOCol = 128;
    static_assert(kOCol + D <= kTileCols && kTiles * kTileCols <= kTmemCols, "tensor memory columns");
};

struct TcBars {
    uint64_t q_full;
    uint64_t k_full[2], k_empty[2], v_full[2], v_empty[2];
    uint64_t s_full[2], p_full[2], o_done[2];  // per query tile
    uint64_t drain;
    uint64_t q_empty;  // per-unit kernel: the pair's last S has read Q
    uint32_t tmem_base;
};

// Waits with every lane of the warp and agrees on the outcome.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity));
}

template <bool B>
struct BoolConst {  // a compile-time flag passed to a generic lambda
    static constexpr bool value = B;
};

constexpr int kRankMaxSeqs = 128;  // batches up to this size can be issued longest-first

// Query rows at positions below this see at most this many keys. In the per-unit kernel
// only the tiles holding such rows give their first chunk's weights to P V as bf16 plus
// the rounding remainder.
constexpr int kPrefillSplitPositions = 64;

// The sequence a CTA with sequence rank z works on: in batches of up to
// kRankMaxSeqs sequences, the z-th by context length (longest first, ties by
// index: with chunks after a long cached context a CTA's work grows with the
// context, so the longest CTAs start first); larger batches in index order.
// Warp 0 ranks the lengths from shared memory; every thread of the CTA calls
// it (it holds a barrier).
__device__ __forceinline__ int prefill_sequence_by_rank(const PrefillParams &pp, int z, int tid) {
    const int S = pp.d.num_seqs;
    if (S > kRankMaxSeqs) return z;
    __shared__ int counts[kRankMaxSeqs];
    __shared__ int chosen;
    if (tid < 32) {
        for (int i = tid; i < S; i += 32) counts[i] = seq_len(pp.d, i, false);
        __syncwarp();
        for (int i = tid; i < S; i += 32) {
            const int ni = counts[i];
            int rank = 0;
            for (int j = 0; j < S; ++j) {
                const int nj = counts[j];
                rank += (nj > ni || (nj == ni && j < i)) ? 1 : 0;
            }
            if (rank == z) chosen = i;
        }
    }
    __syncthreads();
    return chosen;
}

template <int D>
__global__ void __launch_bounds__(TcCfg<D>::kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmv, const PrefillParams pp) {
    using C = TcCfg<D>;
    const DecodeParams &p = pp.d;
    extern __shared__ uint8_t smem_raw[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // Two CTA orders (the grid's shape follows pp.seq_major):
    //  - grid (kv heads, sequences, pairs), the pair index slowest and taken from the
    //    last: every sequence's longest pairs start first and the short ones fill the end;
    //  - grid (kv heads, pairs, sequence rank): one sequence at a time, sequences in
    //    decreasing order of context length, each one's longest pairs first over its kv heads;
    //    a (sequence, kv head)'s pairs start num_kv_heads CTAs apart, so they read its
    //    K/V while it is in L2 without streaming it in lockstep.
    const int h = blockIdx.x;
    int s, pair;
    if (pp.seq_major) {
        pair = gridDim.y - 1 - blockIdx.y;
        s = prefill_sequence_by_rank(pp, blockIdx.z, tid);
    } else {
        s = blockIdx.y;
        pair = gridDim.z - 1 - blockIdx.z;
    }
    const bool flagger = h == 0 && pair == 0;  // one CTA per sequence reports a bad length
    const int g = p.group;
    const int q0 = __ldg(pp.query_start + s), n = __ldg(pp.query_start + s + 1) - q0;
    const int len = seq_len(p, s, tid == 0 && flagger);
    const int tt = pp.tile_tokens;
    if (n < 0 || n > len || n > pp.max_query_len || q0 < 0 || q0 + n > pp.num_queries) {
        if (tid == 0 && flagger) raise_error(PKV_DEVERR_LENGTH);
        return;
    }
    if (pair * C::kTiles * tt >= n) return;
    const int first_pos = len - n;  // position of new token 0
    int t0[C::kTiles], t_end[C::kTiles], nc[C::kTiles];  // per tile: tokens t0 .. t_end - 1, chunks to attend
#pragma unroll
    for (int t = 0; t < C::kTiles; ++t) {
        t0[t] = (pair * C::kTiles + t) * tt;
        t_end[t] = min(n, t0[t] + tt);
        nc[t] = t0[t] < n ? (first_pos + t_end[t] - 1) / C::kKeys + 1 : 0;
    }
    const int nc_all = nc[C::kTiles - 1] > nc[0] ? nc[C::kTiles - 1] : nc[0];
    const int nblk = (len + kBlock - 1) / kBlock;
    const int last_valid = len - (nblk - 1) * kBlock;

    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    TcBars &b = *reinterpret_cast<TcBars *>(base + C::kBarOff);
    if (tid == 0) {
        prefetch_tensormap(&tmq);
        prefetch_tensormap(&tmk);
        prefetch_tensormap(&tmv);
        mbar_init(&b.q_full, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&b.k_full[i], 1);
            mbar_init(&b.k_empty[i], 1);
            mbar_init(&b.v_full[i], 1);
            mbar_init(&b.v_empty[i], 1);
            mbar_init(&b.s_full[i], 1);
            mbar_init(&b.p_full[i], 4);
            mbar_init(&b.o_done[i], 1);
        }
        mbar_init(&b.drain, 1);
        mbar_fence_init();
    }
    if (warp == 1) {
        tmem_alloc(&b.tmem_base, C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = b.tmem_base;
    const uint32_t q_s = smem_u32(base + C::kQOff), k_s = smem_u32(base + C::kKOff);
    const uint32_t v_s = smem_u32(base + C::kVOff);

    if (warp < 4) {
      setmaxnreg_dec<C::kLowRegs>();
      if (warp == 0) {
        // ------------------------------ TMA producer ------------------------------
        if (lane == 0) {
            bool ok = true;
            int qbytes = 0;
#pragma unroll
            for (int t = 0; t < C::kTiles; ++t) qbytes += nc[t] > 0 ? C::kHalves * 128 * g * tt : 0;
            mbar_arrive_expect_tx(&b.q_full, qbytes);
#pragma unroll
            for (int t = 0; t < C::kTiles; ++t)
                if (nc[t] > 0)
                    for (int u = 0; u < C::kHalves; ++u)
                        tma_load_4d(base + C::kQOff + t * C::kQBytes + u * C::kHalfRows, &tmq, 0, u, h * g,
                                    q0 + t0[t], &b.q_full);
            const int32_t *table = p.block_tables + (size_t)s * p.max_blocks_per_seq;
            int issued_k = 0, issued_v = 0;  // chunks whose K / V copies were issued
            for (int j = 0; j < nc_all && ok; ++j) {
                const int st = j & 1;
                if (j >= 2 && !mbar_wait(&b.k_empty[st], ((j - 2) >> 1) & 1)) {
                    ok = false;
                    break;
                }
                // the chunk's blocks: tile row z of the cache view (-1: past the sequence or a bad
                // id, outside the tensor, reads as zeros) and first slot y; the table entries are
                // loaded together so their latencies overlap
                int z[C::kChunkBlocks], y[C::kChunkBlocks];
#pragma unroll
                for (int bi = 0; bi < C::kChunkBlocks; ++bi) {
                    const int blk = j * C::kChunkBlocks + bi;
                    z[bi] = blk < nblk ? __ldg(table + blk) : -1;
                }
#pragma unroll
                for (int bi = 0; bi < C::kChunkBlocks; ++bi) {
                    const int blk = j * C::kChunkBlocks + bi;
                    y[bi] = blk == nblk - 1 ? last_valid - kBlock : 0;
                    if (blk < nblk) {
                        if (z[bi] < 0 || z[bi] >= p.num_blocks) {
                            raise_error(PKV_DEVERR_BLOCK_ID);
                            z[bi] = -1;
                        } else {
                            z[bi] = z[bi] * p.num_kv_heads + h;
                        }
                    }
                }
                // K chunk as [half][128 keys][64]: 8-row groups 1024 bytes apart along the keys
                mbar_arrive_expect_tx(&b.k_full[st], C::kStage);
#pragma unroll
                for (int bi = 0; bi < C::kChunkBlocks; ++bi)
#pragma unroll
                    for (int u = 0; u < C::kHalves; ++u)
                        tma_load_4d(base + C::kKOff + st * C::kStage + u * C::kHalfRows + bi * (kBlock * 128), &tmk,
                                    0, y[bi], u, z[bi], &b.k_full[st]);
                issued_k = j + 1;
                if (j >= 2 && !mbar_wait(&b.v_empty[st], ((j - 2) >> 1) & 1)) {
                    ok = false;
                    break;
                }
                // V chunk as [block][half][16 keys][64]
                mbar_arrive_expect_tx(&b.v_full[st], C::kStage);
#pragma unroll
                for (int bi = 0; bi < C::kChunkBlocks; ++bi)
#pragma unroll
                    for (int u = 0; u < C::kHalves; ++u)
                        tma_load_4d(base + C::kVOff + st * C::kStage + bi * C::kBlockBytes + u * (kBlock * 128),
                                    &tmv, 0, y[bi], u, z[bi], &b.v_full[st]);
                issued_v = j + 1;
            }
            if (!ok) raise_error(PKV_DEVERR_TIMEOUT);
            // no copy may land after the CTA is gone: wait (bounded) for the last one of each stage
            for (int j = max(0, issued_k - 2); j < issued_k; ++j) mbar_wait(&b.k_full[j & 1], (j >> 1) & 1);
            for (int j = max(0, issued_v - 2); j < issued_v; ++j) mbar_wait(&b.v_full[j & 1], (j >> 1) & 1);
            mbar_wait(&b.q_full, 0);
        }
    } else if (warp == 1) {
        // ------------------------------ MMA issuer ------------------------------
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_bf16_f32(C::kRows, C::kKeys, false, false);
            constexpr uint32_t idesc_o = idesc_bf16_f32(C::kRows, D, false, true);
            auto issue_s = [&](int t, int j) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {  // 16 head-dim elements per step
                    const uint32_t off = (kk >> 2) * C::kHalfRows + (kk & 3) * 32;
                    umma_bf16(tmem + t * C::kTileCols, smem_desc_sw128(q_s + t * C::kQBytes + off, 16, 1024),
                              smem_desc_sw128(k_s + (j & 1) * C::kStage + off, 16, 1024), idesc_s, kk > 0);
                }
            };
            auto issue_pv = [&](int t, int j) {
                const bool split = j == 0;  // the first chunk's weights carry their rounding remainder
#pragma unroll
                for (int kk = 0; kk < C::kChunkBlocks; ++kk) {  // 16 keys (one block) per step
                    const uint64_t vd =
                        smem_desc_sw128(v_s + (j & 1) * C::kStage + kk * C::kBlockBytes, kBlock * 128, 1024);
                    // P of keys 16 kk .. 16 kk + 15: columns 32 (kk / 2) + 8 (kk % 2); remainder 16 further
                    const uint32_t pa = tmem + t * C::kTileCols + (kk >> 1) * 32 + (kk & 1) * 8;
                    umma_bf16_tmem_a(tmem + t * C::kTileCols + C::kOCol, pa, vd, idesc_o, j > 0 || kk > 0);
                    if (split) umma_bf16_tmem_a(tmem + t * C::kTileCols + C::kOCol, pa + 16, vd, idesc_o, true);
                }
            };
            bool ok = mbar_wait(&b.q_full, 0) && mbar_wait(&b.k_full[0], 0);
            if (ok) {
                tc_fence_after();
#pragma unroll
                for (int t = 0; t < C::kTiles; ++t)
                    if (nc[t] > 0) {
                        issue_s(t, 0);
                        umma_commit(&b.s_full[t]);
                    }
                umma_commit(&b.k_empty[0]);
            }
            for (int j = 0; ok && j < nc_all; ++j) {
                ok = mbar_wait(&b.v_full[j & 1], (j >> 1) & 1);
                if (ok && j + 1 < nc_all) ok = mbar_wait(&b.k_full[(j + 1) & 1], ((j + 1) >> 1) & 1);
                if (!ok) break;
#pragma unroll
                for (int t = 0; t < C::kTiles; ++t) {
                    if (j >= nc[t]) continue;
                    if (!(ok = mbar_wait(&b.p_full[t], j & 1))) break;
                    tc_fence_after();
                    issue_pv(t, j);
                    if (j + 1 < nc[t]) {
                        issue_s(t, j + 1);
                        umma_commit(&b.s_full[t]);
                    } else {
                        umma_commit(&b.o_done[t]);
                    }
                }
                if (!ok) break;
                umma_commit(&b.v_empty[j & 1]);
                if (j + 1 < nc_all) umma_commit(&b.k_empty[(j + 1) & 1]);
            }
            if (!ok) raise_error(PKV_DEVERR_TIMEOUT);
            // every MMA issued has finished before the tensor memory is released
            umma_commit(&b.drain);
            mbar_wait(&b.drain, 0);
        }
        __syncwarp();
      }
    } else {
        setmaxnreg_inc<C::kHighRegs>();
        // ------------------------------ softmax ------------------------------
        const int t = (warp - 4) >> 2;  // query tile
        const int quad = warp & 3;       // tensor-memory lanes 32 quad .. 32 quad + 31
        const int row = quad * 32 + lane;
        static_assert(C::kTiles == 2, "tile selection below");
        const int ncs = t ? nc[1] : nc[0];           // (selects, not an index: keeps the arrays in registers)
        const int tok0 = t ? t0[1] : t0[0], tok_end = t ? t_end[1] : t_end[0];
        const int rows = ncs > 0 ? (tok_end - tok0) * g : 0;
        const bool row_ok = row < rows;
        const int pos = row_ok ? first_pos + tok0 + row / g : -1;
        const uint32_t cols = tmem + ((uint32_t)(quad * 32) << 16) + t * C::kTileCols;
        const int tile_first = first_pos + tok0;  // the smallest query position of the tile
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        // Scores are kept raw (unscaled): with sl = |scale log2 e| and the sign folded into the scores,
        // x * sl is the log2-domain score, and the max of x gives the max of x * sl.
        const float sl = fabsf(p.scale_log2);
        const float sgn = p.scale_log2 < 0.f ? -1.f : 1.f;
        // Keys of chunk j this row does not see -> -inf. Column kc of a full block holds position
        // 128 j + kc; in the chunk holding the sequence's last block (index lb in the chunk, loaded
        // lo rows early) column kc >= 16 lb holds position 128 j + kc - lo and is a token only
        // from 16 lb + lo on; columns past that block are zeros. So a row at position pos sees
        // columns 0 .. min(P, 16 lb - 1) and 16 lb + lo .. min(P + lo, 16 lb + 15), P = pos - 128 j.
        auto mask = [&](float (&v)[4][32], int j) {
            const int P = pos - j * C::kKeys;
            const int lb = nblk - 1 - j * C::kChunkBlocks;
            if (lb >= C::kChunkBlocks) {
#pragma unroll
                for (int q = 0; q < 4; ++q)
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[q][e] = q * 32 + e <= P ? v[q][e] : -INFINITY;
            } else {
                const int lo = kBlock - last_valid;
                const int a_end = min(P, lb * kBlock - 1);
                const int b_lo = lb * kBlock + lo, b_hi = min(P + lo, lb * kBlock + kBlock - 1);
#pragma unroll
                for (int q = 0; q < 4; ++q)
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const int kc = q * 32 + e;
                        v[q][e] = (kc <= a_end || (kc >= b_lo && kc <= b_hi)) ? v[q][e] : -INFINITY;
                    }
            }
        };
        for (int j = 0; j < ncs; ++j) {
            if (!(ok = warp_wait(&b.s_full[t], j & 1))) break;
            tc_fence_after();
            // the whole row of S_t in registers (one tensor-memory round trip)
            float x[4][32];
#pragma unroll
            for (int q = 0; q < 4; ++q) tmem_ld32(cols + q * 32, x[q]);
            tmem_wait_ld();
            if (sgn < 0.f) {
#pragma unroll
                for (int q = 0; q < 4; ++q)
#pragma unroll
                    for (int e = 0; e < 32; ++e) x[q][e] = -x[q][e];
            }
            // only chunks holding the end of the sequence, or keys past the tile's first query, need masks
            const bool plain = (j + 1) * C::kChunkBlocks < nblk && (j + 1) * C::kKeys - 1 <= tile_first;
            if (!plain) mask(x, j);
            float mxs[8];  // independent partial maxima (a single chain would be 128 dependent steps)
#pragma unroll
            for (int i = 0; i < 8; ++i) mxs[i] = -INFINITY;
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
                for (int e = 0; e < 32; e += 2) mxs[(e >> 1) & 7] = max3f(mxs[(e >> 1) & 7], x[q][e], x[q][e + 1]);
            const float mx = fmaxf(fmaxf(fmaxf(mxs[0], mxs[1]), fmaxf(mxs[2], mxs[3])),
                                   fmaxf(fmaxf(mxs[4], mxs[5]), fmaxf(mxs[6], mxs[7])));
            const float m_new = fmaxf(m, mx * sl);
            const bool move = m_new > m + 8.f;
            const float m_use = move ? m_new : m;
            const float ms = m_use == -INFINITY ? 0.f : m_use;
            const float alpha = ex2_approx(m - ms);
            // this tile's O is quiescent here (P V of the previous chunk ran before S of this one)
            if (j > 0 && __any_sync(0xffffffffu, move && m != -INFINITY)) {
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    float o[32];
                    tmem_ld32(cols + C::kOCol + c * 32, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] *= alpha;
                    tmem_st32(cols + C::kOCol + c * 32, o);
                }
            }
            m = m_use;
            // P = 2^(x sl - reference max) in bf16 over each quarter's own score columns:
            // keys 32 q + 2 i, + 1 at column 32 q + i, their rounding remainders at + 16.
            // The row sum takes the unrounded weights: the first chunk's P (hi + lo) matches
            // them to 2^-16, later chunks' rounding errors average out over the keys.
            const bool split = j == 0;
            const uint64_t sl2 = pack_f2(sl, sl), nms2 = pack_f2(-ms, -ms);
            uint64_t rss[4];  // independent partial sums, two lanes each
#pragma unroll
            for (int i = 0; i < 4; ++i) rss[i] = pack_f2(0.f, 0.f);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint32_t hi[16], lo[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float a0, a1;
                    unpack_f2(fma_f2(pack_f2(x[q][2 * i], x[q][2 * i + 1]), sl2, nms2), a0, a1);
                    const float e0 = ex2_approx(a0), e1 = ex2_approx(a1);
                    rss[i & 3] = add_f2(rss[i & 3], pack_f2(e0, e1));
                    const __nv_bfloat162 ph = __floats2bfloat162_rn(e0, e1);
                    hi[i] = *reinterpret_cast<const uint32_t *>(&ph);
                    if (split) {
                        const float2 fh = __bfloat1622float2(ph);
                        const __nv_bfloat162 pl = __floats2bfloat162_rn(e0 - fh.x, e1 - fh.y);
                        lo[i] = *reinterpret_cast<const uint32_t *>(&pl);
                    }
                }
                tmem_st16(cols + q * 32, hi);
                if (split) tmem_st16(cols + q * 32 + 16, lo);
            }
            tmem_wait_st();
            float rs;
            {
                float r[8];
#pragma unroll
                for (int i = 0; i < 4; ++i) unpack_f2(rss[i], r[2 * i], r[2 * i + 1]);
                rs = ((r[0] + r[1]) + (r[2] + r[3])) + ((r[4] + r[5]) + (r[6] + r[7]));
            }
            l = l * alpha + rs;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&b.p_full[t]);
        }
        if (ncs > 0) {
            if (ok) ok = warp_wait(&b.o_done[t], 0);
            if (!ok) {
                raise_error(PKV_DEVERR_TIMEOUT);
            } else {
                tc_fence_after();
                const float inv = l > 0.f ? 1.f / l : 0.f;
                __nv_bfloat16 *dst =
                    static_cast<__nv_bfloat16 *>(p.out) +
                    ((size_t)(q0 + tok0 + (row_ok ? row / g : 0)) * p.num_q_heads + h * g + row % g) * D;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    float o[32];
                    tmem_ld32(cols + C::kOCol + c * 32, o);
                    tmem_wait_ld();
                    if (row_ok) {
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            uint32_t w[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const __nv_bfloat162 v2 = __floats2bfloat162_rn(o[q * 8 + 2 * e] * inv,
                                                                                o[q * 8 + 2 * e + 1] * inv);
                                w[e] = *reinterpret_cast<const uint32_t *>(&v2);
                            }
                            *reinterpret_cast<uint4 *>(dst + c * 32 + q * 8) = make_uint4(w[0], w[1], w[2], w[3]);
                        }
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}


// The same attention with one CTA per (sequence, kv head) taking all its pairs, longest
// first: grid (kv heads, sequence rank). For whole prompts in batches with many such units:
// the CTA's set-up (tensor-memory allocation, barriers) is paid once, and the next pair's Q
// and first K/V chunk load while the current pair finishes. The roles are those of
// prefill_tc_kernel, each looping over the pairs; barrier phases run on across pairs (a
// K/V ring position over all the CTA's chunks, per-tile S / P and O phase counts), and a
// q_empty barrier lets the next pair's Q land only once the last S of the pair has read Q.
template <int D>
__global__ void __launch_bounds__(TcCfg<D>::kThreads, 1)
    prefill_tc_units_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmv, const PrefillParams pp) {
    using C = TcCfg<D>;
    const DecodeParams &p = pp.d;
    extern __shared__ uint8_t smem_raw[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.x;
    const int s = prefill_sequence_by_rank(pp, blockIdx.y, tid);
    const bool flagger = h == 0;  // one CTA per sequence reports a bad length
    const int g = p.group;
    const int q0 = __ldg(pp.query_start + s), n = __ldg(pp.query_start + s + 1) - q0;
    const int len = seq_len(p, s, tid == 0 && flagger);
    const int tt = pp.tile_tokens;
    if (n < 0 || n > len || n > pp.max_query_len || q0 < 0 || q0 + n > pp.num_queries) {
        if (tid == 0 && flagger) raise_error(PKV_DEVERR_LENGTH);
        return;
    }
    const int npairs = (n + C::kTiles * tt - 1) / (C::kTiles * tt);  // pair_hi - it for it < npairs
    const int pair_hi = npairs - 1;
    if (npairs == 0) return;
    const int first_pos = len - n;  // position of new token 0
    // Tiles of the it-th pair: tokens t0 .. t_end - 1 and the chunks they attend; returns
    // the pair's chunk count.
    auto pair_tiles = [&](int it, int (&t0)[C::kTiles], int (&t_end)[C::kTiles], int (&nc)[C::kTiles]) -> int {
        const int pair = pair_hi - it;
#pragma unroll
        for (int t = 0; t < C::kTiles; ++t) {
            t0[t] = (pair * C::kTiles + t) * tt;
            t_end[t] = min(n, t0[t] + tt);
            nc[t] = t0[t] < n ? (first_pos + t_end[t] - 1) / C::kKeys + 1 : 0;
        }
        return nc[C::kTiles - 1] > nc[0] ? nc[C::kTiles - 1] : nc[0];
    };
    // The same, chunk counts only (the MMA thread needs no more).
    auto pair_chunks = [&](int it, int (&nc)[C::kTiles]) -> int {
        const int pair = pair_hi - it;
#pragma unroll
        for (int t = 0; t < C::kTiles; ++t) {
            const int a = (pair * C::kTiles + t) * tt;
            nc[t] = a < n ? (first_pos + min(n, a + tt) - 1) / C::kKeys + 1 : 0;
        }
        return nc[C::kTiles - 1] > nc[0] ? nc[C::kTiles - 1] : nc[0];
    };
    const int nblk = (len + kBlock - 1) / kBlock;
    const int last_valid = len - (nblk - 1) * kBlock;

    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    TcBars &b = *reinterpret_cast<TcBars *>(base + C::kBarOff);
    if (tid == 0) {
        prefetch_tensormap(&tmq);
        prefetch_tensormap(&tmk);
        prefetch_tensormap(&tmv);
        mbar_init(&b.q_full, 1);
        mbar_init(&b.q_empty, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&b.k_full[i], 1);
            mbar_init(&b.k_empty[i], 1);
            mbar_init(&b.v_full[i], 1);
            mbar_init(&b.v_empty[i], 1);
            mbar_init(&b.s_full[i], 1);
            mbar_init(&b.p_full[i], 4);
            mbar_init(&b.o_done[i], 1);
        }
        mbar_init(&b.drain, 1);
        mbar_fence_init();
    }
    if (warp == 1) {
        tmem_alloc(&b.tmem_base, C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = b.tmem_base;
    const uint32_t q_s = smem_u32(base + C::kQOff), k_s = smem_u32(base + C::kKOff);
    const uint32_t v_s = smem_u32(base + C::kVOff);

    if (warp < 4) {
      setmaxnreg_dec<C::kLowRegs>();
      if (warp == 0) {
        // ------------------------------ TMA producer ------------------------------
        if (lane == 0) {
            bool ok = true;
            const int32_t *table = p.block_tables + (size_t)s * p.max_blocks_per_seq;
            int issued_k = 0, issued_v = 0, issued_q = 0;  // K / V chunks (all pairs) and Q tiles issued
            for (int it = 0; it < npairs && ok; ++it) {
            int t0[C::kTiles], t_end[C::kTiles], nc[C::kTiles];
            const int nc_all = pair_tiles(it, t0, t_end, nc);
            // the previous pair's last S has read Q before this pair's Q lands there
            if (it > 0 && !mbar_wait(&b.q_empty, (it - 1) & 1)) {
                ok = false;
                break;
            }
            int qbytes = 0;
#pragma unroll
            for (int t = 0; t < C::kTiles; ++t) qbytes += nc[t] > 0 ? C::kHalves * 128 * g * tt : 0;
            mbar_arrive_expect_tx(&b.q_full, qbytes);
#pragma unroll
            for (int t = 0; t < C::kTiles; ++t)
                if (nc[t] > 0)
                    for (int u = 0; u < C::kHalves; ++u)
                        tma_load_4d(base + C::kQOff + t * C::kQBytes + u * C::kHalfRows, &tmq, 0, u, h * g,
                                    q0 + t0[t], &b.q_full);
            issued_q = it + 1;
            for (int j = 0; j < nc_all && ok; ++j) {
                const int gj = issued_k;  // ring position over all the CTA's chunks
                const int st = gj & 1;
                if (gj >= 2 && !mbar_wait(&b.k_empty[st], ((gj - 2) >> 1) & 1)) {
                    ok = false;
                    break;
                }
                // the chunk's blocks: tile row z of the cache view (-1: past the sequence or a bad
                // id, outside the tensor, reads as zeros) and first slot y; the table entries are
                // loaded together so their latencies overlap
                int z[C::kChunkBlocks], y[C::kChunkBlocks];
#pragma unroll
                for (int bi = 0; bi < C::kChunkBlocks; ++bi) {
                    const int blk = j * C::kChunkBlocks + bi;
                    z[bi] = blk < nblk ? __ldg(table + blk) : -1;
                }
#pragma unroll
                for (int bi = 0; bi < C::kChunkBlocks; ++bi) {
                    const int blk = j * C::kChunkBlocks + bi;
                    y[bi] = blk == nblk - 1 ? last_valid - kBlock : 0;
                    if (blk < nblk) {
                        if (z[bi] < 0 || z[bi] >= p.num_blocks) {
                            raise_error(PKV_DEVERR_BLOCK_ID);
                            z[bi] = -1;
                        } else {
                            z[bi] = z[bi] * p.num_kv_heads + h;
                        }
                    }
                }
                // K chunk as [half][128 keys][64]: 8-row groups 1024 bytes apart along the keys
                mbar_arrive_expect_tx(&b.k_full[st], C::kStage);
#pragma unroll
                for (int bi = 0; bi < C::kChunkBlocks; ++bi)
#pragma unroll
                    for (int u = 0; u < C::kHalves; ++u)
                        tma_load_4d(base + C::kKOff + st * C::kStage + u * C::kHalfRows + bi * (kBlock * 128), &tmk,
                                    0, y[bi], u, z[bi], &b.k_full[st]);
                issued_k = gj + 1;
                if (gj >= 2 && !mbar_wait(&b.v_empty[st], ((gj - 2) >> 1) & 1)) {
                    ok = false;
                    break;
                }
                // V chunk as [block][half][16 keys][64]
                mbar_arrive_expect_tx(&b.v_full[st], C::kStage);
#pragma unroll
                for (int bi = 0; bi < C::kChunkBlocks; ++bi)
#pragma unroll
                    for (int u = 0; u < C::kHalves; ++u)
                        tma_load_4d(base + C::kVOff + st * C::kStage + bi * C::kBlockBytes + u * (kBlock * 128),
                                    &tmv, 0, y[bi], u, z[bi], &b.v_full[st]);
                issued_v = gj + 1;
            }
            }
            if (!ok) raise_error(PKV_DEVERR_TIMEOUT);
            // no copy may land after the CTA is gone: wait (bounded) for the last one of each stage
            for (int j = max(0, issued_k - 2); j < issued_k; ++j) mbar_wait(&b.k_full[j & 1], (j >> 1) & 1);
            for (int j = max(0, issued_v - 2); j < issued_v; ++j) mbar_wait(&b.v_full[j & 1], (j >> 1) & 1);
            if (issued_q > 0) mbar_wait(&b.q_full, (issued_q - 1) & 1);
        }
    } else if (warp == 1) {
        // ------------------------------ MMA issuer ------------------------------
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_bf16_f32(C::kRows, C::kKeys, false, false);
            constexpr uint32_t idesc_o = idesc_bf16_f32(C::kRows, D, false, true);
            // S of tile t from the K chunk in ring position gj
            auto issue_s = [&](int t, int gj) {
                // (opaque bases: the descriptors are built at the issue, not hoisted and held in
                // registers across the pair loop)
                uint32_t qb = q_s + t * C::kQBytes, kb = k_s + (gj & 1) * C::kStage;
                asm volatile("" : "+r"(qb), "+r"(kb));
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {  // 16 head-dim elements per step
                    const uint32_t off = (kk >> 2) * C::kHalfRows + (kk & 3) * 32;
                    umma_bf16(tmem + t * C::kTileCols, smem_desc_sw128(qb + off, 16, 1024),
                              smem_desc_sw128(kb + off, 16, 1024), idesc_s, kk > 0);
                }
            };
            // O of tile t += P V, chunk j of the pair from the V chunk in ring position gj
            auto issue_pv = [&](int t, int j, int gj, bool split_tile) {
                // the first chunk's weights carry their rounding remainder in tiles with rows that see few keys
                const bool split = j == 0 && split_tile;
                uint32_t vb = v_s + (gj & 1) * C::kStage;
                asm volatile("" : "+r"(vb));
#pragma unroll
                for (int kk = 0; kk < C::kChunkBlocks; ++kk) {  // 16 keys (one block) per step
                    const uint64_t vd = smem_desc_sw128(vb + kk * C::kBlockBytes, kBlock * 128, 1024);
                    // P of keys 16 kk .. 16 kk + 15: columns 32 (kk / 2) + 8 (kk % 2); remainder 16 further
                    const uint32_t pa = tmem + t * C::kTileCols + (kk >> 1) * 32 + (kk & 1) * 8;
                    umma_bf16_tmem_a(tmem + t * C::kTileCols + C::kOCol, pa, vd, idesc_o, j > 0 || kk > 0);
                    if (split) umma_bf16_tmem_a(tmem + t * C::kTileCols + C::kOCol, pa + 16, vd, idesc_o, true);
                }
            };
            bool ok = true;
            int kv = 0;                // ring position of the pair's first chunk
            int cs[C::kTiles] = {};    // per tile: chunks of the earlier pairs (S / P phases)
            for (int it = 0; it < npairs && ok; ++it) {
                int nc[C::kTiles];
                const int nc_all = pair_chunks(it, nc);
                int split_tiles = 0;  // tiles whose first chunk is split, one bit each
#pragma unroll
                for (int t = 0; t < C::kTiles; ++t)
                    split_tiles |= (first_pos + ((pair_hi - it) * C::kTiles + t) * tt < kPrefillSplitPositions) << t;
                ok = mbar_wait(&b.q_full, it & 1) && mbar_wait(&b.k_full[kv & 1], (kv >> 1) & 1);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int t = 0; t < C::kTiles; ++t)
                    if (nc[t] > 0) {
                        issue_s(t, kv);
                        umma_commit(&b.s_full[t]);
                    }
                umma_commit(&b.k_empty[kv & 1]);
                if (nc_all == 1) umma_commit(&b.q_empty);  // the pair's last S has been issued
                for (int j = 0; ok && j < nc_all; ++j) {
                    const int gj = kv + j;
                    ok = mbar_wait(&b.v_full[gj & 1], (gj >> 1) & 1);
                    if (ok && j + 1 < nc_all) ok = mbar_wait(&b.k_full[(gj + 1) & 1], ((gj + 1) >> 1) & 1);
                    if (!ok) break;
#pragma unroll
                    for (int t = 0; t < C::kTiles; ++t) {
                        if (j >= nc[t]) continue;
                        if (!(ok = mbar_wait(&b.p_full[t], (cs[t] + j) & 1))) break;
                        tc_fence_after();
                        issue_pv(t, j, gj, (split_tiles >> t) & 1);
                        if (j + 1 < nc[t]) {
                            issue_s(t, gj + 1);
                            umma_commit(&b.s_full[t]);
                        } else {
                            umma_commit(&b.o_done[t]);
                        }
                    }
                    if (!ok) break;
                    umma_commit(&b.v_empty[gj & 1]);
                    if (j + 1 < nc_all) umma_commit(&b.k_empty[(gj + 1) & 1]);
                    if (j + 2 == nc_all) umma_commit(&b.q_empty);  // the pair's last S has been issued
                }
#pragma unroll
                for (int t = 0; t < C::kTiles; ++t) cs[t] += nc[t];
                kv += nc_all;
            }
            if (!ok) raise_error(PKV_DEVERR_TIMEOUT);
            // every MMA issued has finished before the tensor memory is released
            umma_commit(&b.drain);
            mbar_wait(&b.drain, 0);
        }
        __syncwarp();
      }
    } else {
        setmaxnreg_inc<C::kHighRegs>();
        // ------------------------------ softmax ------------------------------
        const int t = (warp - 4) >> 2;  // query tile
        const int quad = warp & 3;       // tensor-memory lanes 32 quad .. 32 quad + 31
        const int row = quad * 32 + lane;
        static_assert(C::kTiles == 2, "tile selection below");
        const uint32_t cols = tmem + ((uint32_t)(quad * 32) << 16) + t * C::kTileCols;
        int pos = -1;  // this row's query position in the current pair (-1: no row)
        bool ok = true;
        // Scores are kept raw (unscaled): with sl = |scale log2 e| and the sign folded into the scores,
        // x * sl is the log2-domain score, and the max of x gives the max of x * sl.
        const float sl = fabsf(p.scale_log2);
        const float sgn = p.scale_log2 < 0.f ? -1.f : 1.f;
        // Keys of chunk j this row does not see -> -inf. Column kc of a full block holds position
        // 128 j + kc; in the chunk holding the sequence's last block (index lb in the chunk, loaded
        // lo rows early) column kc >= 16 lb holds position 128 j + kc - lo and is a token only
        // from 16 lb + lo on; columns past that block are zeros. So a row at position pos sees
        // columns 0 .. min(P, 16 lb - 1) and 16 lb + lo .. min(P + lo, 16 lb + 15), P = pos - 128 j.
        auto mask = [&](float (&v)[4][32], int j) {
            const int P = pos - j * C::kKeys;
            const int lb = nblk - 1 - j * C::kChunkBlocks;
            if (lb >= C::kChunkBlocks) {
#pragma unroll
                for (int q = 0; q < 4; ++q)
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[q][e] = q * 32 + e <= P ? v[q][e] : -INFINITY;
            } else {
                const int lo = kBlock - last_valid;
                const int a_end = min(P, lb * kBlock - 1);
                const int b_lo = lb * kBlock + lo, b_hi = min(P + lo, lb * kBlock + kBlock - 1);
#pragma unroll
                for (int q = 0; q < 4; ++q)
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const int kc = q * 32 + e;
                        v[q][e] = (kc <= a_end || (kc >= b_lo && kc <= b_hi)) ? v[q][e] : -INFINITY;
                    }
            }
        };
        int cs = 0, od = 0;  // this tile's chunks and outputs in the earlier pairs (S / P and O phases)
        for (int it = 0; it < npairs && ok; ++it) {
        int t0[C::kTiles], t_end[C::kTiles], nc[C::kTiles];
        pair_tiles(it, t0, t_end, nc);
        const int ncs = t ? nc[1] : nc[0];           // (selects, not an index: keeps the arrays in registers)
        const int tok0 = t ? t0[1] : t0[0], tok_end = t ? t_end[1] : t_end[0];
        const int rows = ncs > 0 ? (tok_end - tok0) * g : 0;
        const bool row_ok = row < rows;
        pos = row_ok ? first_pos + tok0 + row / g : -1;
        const int tile_first = first_pos + tok0;  // the smallest query position of the tile
        const bool split_tile = tile_first < kPrefillSplitPositions;  // its rows include some that see few keys
        float m = -INFINITY, l = 0.f;
        for (int j = 0; j < ncs; ++j) {
            if (!(ok = warp_wait(&b.s_full[t], (cs + j) & 1))) break;
            tc_fence_after();
            // the whole row of S_t in registers (one tensor-memory round trip)
            float x[4][32];
#pragma unroll
            for (int q = 0; q < 4; ++q) tmem_ld32(cols + q * 32, x[q]);
            tmem_wait_ld();
            if (sgn < 0.f) {
#pragma unroll
                for (int q = 0; q < 4; ++q)
#pragma unroll
                    for (int e = 0; e < 32; ++e) x[q][e] = -x[q][e];
            }
            // only chunks holding the end of the sequence, or keys past the tile's first query, need masks
            const bool plain = (j + 1) * C::kChunkBlocks < nblk && (j + 1) * C::kKeys - 1 <= tile_first;
            if (!plain) mask(x, j);
            float mxs[8];  // independent partial maxima (a single chain would be 128 dependent steps)
#pragma unroll
            for (int i = 0; i < 8; ++i) mxs[i] = -INFINITY;
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
                for (int e = 0; e < 32; e += 2) mxs[(e >> 1) & 7] = max3f(mxs[(e >> 1) & 7], x[q][e], x[q][e + 1]);
            const float mx = fmaxf(fmaxf(fmaxf(mxs[0], mxs[1]), fmaxf(mxs[2], mxs[3])),
                                   fmaxf(fmaxf(mxs[4], mxs[5]), fmaxf(mxs[6], mxs[7])));
            const float m_new = fmaxf(m, mx * sl);
            const bool move = m_new > m + 8.f;
            const float m_use = move ? m_new : m;
            const float ms = m_use == -INFINITY ? 0.f : m_use;
            const float alpha = ex2_approx(m - ms);
            // this tile's O is quiescent here (P V of the previous chunk ran before S of this one)
            if (j > 0 && __any_sync(0xffffffffu, move && m != -INFINITY)) {
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    float o[32];
                    tmem_ld32(cols + C::kOCol + c * 32, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] *= alpha;
                    tmem_st32(cols + C::kOCol + c * 32, o);
                }
            }
            m = m_use;
            // P = 2^(x sl - reference max) in bf16 over each quarter's own score columns:
            // keys 32 q + 2 i, + 1 at column 32 q + i, their rounding remainders at + 16.
            // The row sum takes the unrounded weights: the first chunk's P (hi + lo) matches
            // them to 2^-16, later chunks' rounding errors average out over the keys.
            // (compiled twice: the first chunk's instance with the remainders, the others' without,
            // so the common chunk's code carries none of the split's instructions or registers)
            auto write_p = [&](auto split_c) -> float {
                constexpr bool split = decltype(split_c)::value;
                const uint64_t sl2 = pack_f2(sl, sl), nms2 = pack_f2(-ms, -ms);
                uint64_t rss[4];  // independent partial sums, two lanes each
#pragma unroll
                for (int i = 0; i < 4; ++i) rss[i] = pack_f2(0.f, 0.f);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint32_t hi[16], lo[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        float a0, a1;
                        unpack_f2(fma_f2(pack_f2(x[q][2 * i], x[q][2 * i + 1]), sl2, nms2), a0, a1);
                        const float e0 = ex2_approx(a0), e1 = ex2_approx(a1);
                        rss[i & 3] = add_f2(rss[i & 3], pack_f2(e0, e1));
                        const __nv_bfloat162 ph = __floats2bfloat162_rn(e0, e1);
                        hi[i] = *reinterpret_cast<const uint32_t *>(&ph);
                        if constexpr (split) {
                            const float2 fh = __bfloat1622float2(ph);
                            const __nv_bfloat162 pl = __floats2bfloat162_rn(e0 - fh.x, e1 - fh.y);
                            lo[i] = *reinterpret_cast<const uint32_t *>(&pl);
                        }
                    }
                    tmem_st16(cols + q * 32, hi);
                    if constexpr (split) tmem_st16(cols + q * 32 + 16, lo);
                }
                tmem_wait_st();
                float r[8];
#pragma unroll
                for (int i = 0; i < 4; ++i) unpack_f2(rss[i], r[2 * i], r[2 * i + 1]);
                return ((r[0] + r[1]) + (r[2] + r[3])) + ((r[4] + r[5]) + (r[6] + r[7]));
            };
            const float rs = j == 0 && split_tile ? write_p(BoolConst<true>{}) : write_p(BoolConst<false>{});
            l = l * alpha + rs;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&b.p_full[t]);
        }
        if (ncs > 0) {
            if (ok) ok = warp_wait(&b.o_done[t], od & 1);
            ++od;
            if (!ok) {
                raise_error(PKV_DEVERR_TIMEOUT);
            } else {
                tc_fence_after();
                const float inv = l > 0.f ? 1.f / l : 0.f;
                __nv_bfloat16 *dst =
                    static_cast<__nv_bfloat16 *>(p.out) +
                    ((size_t)(q0 + tok0 + (row_ok ? row / g : 0)) * p.num_q_heads + h * g + row % g) * D;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    float o[32];
                    tmem_ld32(cols + C::kOCol + c * 32, o);
                    tmem_wait_ld();
                    if (row_ok) {
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            uint32_t w[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const __nv_bfloat162 v2 = __floats2bfloat162_rn(o[q * 8 + 2 * e] * inv,
                                                                                o[q * 8 + 2 * e + 1] * inv);
                                w[e] = *reinterpret_cast<const uint32_t *>(&v2);
                            }
                            *reinterpret_cast<uint4 *>(dst + c * 32 + q * 8) = make_uint4(w[0], w[1], w[2], w[3]);
                        }
                    }
                }
            }
        }
        cs += ncs;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

}  // namespace pkv
