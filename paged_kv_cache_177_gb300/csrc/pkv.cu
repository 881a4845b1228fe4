// pkv.cu -- host side of the C ABI declared in include/pagedkv.h: argument
// checks, split-context planning, TMA descriptor encoding and launches.
// The library never allocates device memory and never synchronises, except
// pkv_device_error(), which is documented as synchronous.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <unordered_set>

#include "pagedkv.h"
#include "pkv_kernels.cuh"
#include "pkv_prefill_tc.cuh"

namespace {

constexpr int kVersion = 100;          // 0.1.0
constexpr int kDefaultPartition = 512; // tokens per split-context partition (32 blocks)
constexpr int kMaxParts = 8192;        // partitions per sequence the reduce kernel handles
// Launch shapes (compile-time; -D overrides are for tuning sweeps).
#ifndef PKV_GRID_STAGES
#define PKV_GRID_STAGES 8
#endif
#ifndef PKV_GRID_CONSUMERS
#define PKV_GRID_CONSUMERS 4
#endif
#ifndef PKV_PERSIST_WARPS
#define PKV_PERSIST_WARPS 12
#endif
#ifndef PKV_PERSIST_STAGES_D128
#define PKV_PERSIST_STAGES_D128 1
#endif
#ifndef PKV_PERSIST_STAGES_D64
#define PKV_PERSIST_STAGES_D64 2
#endif
#ifndef PKV_MHA_CUDA_CORES
#define PKV_MHA_CUDA_CORES 1
#endif
constexpr int kNstage = PKV_GRID_STAGES;
constexpr bool kMhaCudaCores = PKV_MHA_CUDA_CORES != 0;  // g = 1 on the CUDA cores (persistent kernel)
#ifndef PKV_PREFILL_UNITS
#define PKV_PREFILL_UNITS 1
#endif
constexpr bool kPrefillUnits = PKV_PREFILL_UNITS != 0;  // prefill: one CTA per (sequence, kv head) when many

constexpr int kNcw = PKV_GRID_CONSUMERS;
// persistent bf16 kernel: one CTA of kPersistWarps warps per SM
constexpr int kPersistWarps = PKV_PERSIST_WARPS;
constexpr int kPersistMaxCtas = 160;     // sizes the workspace; GB300 has 152 SMs
#ifndef PKV_PERSIST_MAX_SEQS
#define PKV_PERSIST_MAX_SEQS 8192
#endif
constexpr int kPersistMaxSeqs = PKV_PERSIST_MAX_SEQS;  // block-count prefix sums live in shared memory
constexpr size_t kSmemLimit = 232448;    // 227 KiB per CTA

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int elem_bytes(pkv_dtype dt) { return dt == PKV_BF16 ? 2 : 4; }

bool dtype_ok(pkv_dtype dt) { return dt == PKV_BF16 || dt == PKV_F32; }

// The storage type of q and the caches for a decode dtype (PKV_BF16_OUT_F32
// reads bf16 and writes fp32).
pkv_dtype input_dtype(pkv_dtype dt) { return dt == PKV_BF16_OUT_F32 ? PKV_BF16 : dt; }

int check_launch() {
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

// Launches `kern` with programmatic stream serialisation: it may start while
// the previous kernel of the stream runs (that kernel's blocks call
// pdl_trigger; the new kernel calls pdl_wait before reading what it writes).
template <typename... Params, typename... Args>
int launch_pdl(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...) == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

// cuTensorMapEncodeTiled from the driver, fetched through the runtime so the
// library does not link libcuda directly.
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// 4-D view of a cache that makes one TMA box of each (block, kv head) tile:
// x = element within a 64-element (128-byte) half row, y = slot (16, stride
// one row), z = which half of the row (head_dim / 64, stride 128 bytes),
// w = (block * Hkv + head) tile. The box {64, 16, head_dim / 64, 1} is the
// whole contiguous tile, landing in shared memory as [half][slot][64] with
// the 128-byte swizzle on each 128-byte row. Loading from y = valid - 16
// makes TMA zero-fill the rows before the tile start: that is how the last
// block of a sequence arrives with its slots past the end already zero.
int encode_cache_map(CUtensorMap *map, const void *cache, int num_blocks, int num_kv_heads, int head_dim,
                     bool one_half = false) {
    auto fn = encode_fn();
    if (!fn) return PKV_ERR_CUDA;
    cuuint64_t dims[4] = {64, 16, (cuuint64_t)head_dim / 64, (cuuint64_t)num_blocks * num_kv_heads};
    cuuint64_t strides[3] = {(cuuint64_t)head_dim * 2, 128, (cuuint64_t)head_dim * 2 * 16};
    cuuint32_t box[4] = {64, 16, one_half ? 1u : (cuuint32_t)head_dim / 64, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(cache), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PKV_OK : PKV_ERR_CUDA;
}

// (one_half: a box of one 64-element half of the 16 slots' rows, 2 KiB, so a
// caller can place the halves of consecutive blocks apart.)

// The same view of an fp32 cache: x = element within a 32-element (128-byte) quarter
// or half row, z = which one (head_dim / 32). The box {32, 16, head_dim / 32, 1} is the
// whole tile, landing as [sub-tile][slot][32] with the 128-byte swizzle.
int encode_cache_map_f32(CUtensorMap *map, const void *cache, int num_blocks, int num_kv_heads, int head_dim) {
    auto fn = encode_fn();
    if (!fn) return PKV_ERR_CUDA;
    cuuint64_t dims[4] = {32, 16, (cuuint64_t)head_dim / 32, (cuuint64_t)num_blocks * num_kv_heads};
    cuuint64_t strides[3] = {(cuuint64_t)head_dim * 4, 128, (cuuint64_t)head_dim * 4 * 16};
    cuuint32_t box[4] = {32, 16, (cuuint32_t)head_dim / 32, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<void *>(cache), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PKV_OK : PKV_ERR_CUDA;
}

// 4-D view of q [T][Hq][D] for the tensor-core prefill: x = element within a
// 64-element half row, y = half, z = query head, w = query row (token). The
// box {64, 1, g, tokens} lands one half of a (token, head) tile as rows
// token * g + head of 128 bytes, with the 128-byte swizzle.
int encode_q_map(CUtensorMap *map, const void *q, int num_queries, int num_q_heads, int head_dim, int g,
                 int tokens) {
    auto fn = encode_fn();
    if (!fn) return PKV_ERR_CUDA;
    cuuint64_t dims[4] = {64, (cuuint64_t)head_dim / 64, (cuuint64_t)num_q_heads, (cuuint64_t)num_queries};
    cuuint64_t strides[3] = {128, (cuuint64_t)head_dim * 2, (cuuint64_t)num_q_heads * head_dim * 2};
    cuuint32_t box[4] = {64, 1, (cuuint32_t)g, (cuuint32_t)tokens};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(q), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PKV_OK : PKV_ERR_CUDA;
}

int max_parts_for(int max_context_len, int part_tokens) {
    if (max_context_len <= 0) return 1;
    return (max_context_len + part_tokens - 1) / part_tokens;
}

template <int D, int NT, typename OutT, class WA = pkv::WarpAttn<D, NT>>
int launch_bf16(const CUtensorMap &tmk, const CUtensorMap &tmv, const pkv::DecodeParams &p, dim3 grid,
                cudaStream_t st, bool pdl = false) {
    using C = pkv::Bf16Cfg<D, NT, kNstage, kNcw>;
    auto kern = pkv::decode_bf16_kernel<D, NT, kNstage, kNcw, OutT, WA>;
    static thread_local int configured_device = -1;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    if (configured_device != dev) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem) != cudaSuccess)
            return PKV_ERR_CUDA;
        configured_device = dev;
    }
    if (pdl) return launch_pdl(kern, grid, dim3(C::kThreads), C::kSmem, st, tmk, tmv, p);
    kern<<<grid, C::kThreads, C::kSmem, st>>>(tmk, tmv, p);
    return check_launch();
}


// fp32 caches: the staged kernel with the query-head bound GMAX >= g, four stages (a
// stage is 16 KiB at d = 128).
#ifndef PKV_F32_STAGES
#define PKV_F32_STAGES 4
#endif
#ifndef PKV_F32_NCW
#define PKV_F32_NCW 4
#endif
constexpr int kF32Stages = PKV_F32_STAGES, kF32Ncw = PKV_F32_NCW;

template <int D, int GMAX>
int launch_f32_staged(const CUtensorMap &tmk, const CUtensorMap &tmv, const pkv::DecodeParams &p, dim3 grid,
                      cudaStream_t st, bool pdl) {
    using C = pkv::F32Cfg<D, GMAX, kF32Stages, kF32Ncw>;
    static_assert(C::kSmem <= (int)kSmemLimit, "shared memory");
    auto kern = pkv::decode_f32_staged_kernel<D, GMAX, kF32Stages, kF32Ncw>;
    static thread_local int configured_device = -1;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    if (configured_device != dev) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem) != cudaSuccess)
            return PKV_ERR_CUDA;
        configured_device = dev;
    }
    if (pdl) return launch_pdl(kern, grid, dim3(C::kThreads), C::kSmem, st, tmk, tmv, p);
    kern<<<grid, C::kThreads, C::kSmem, st>>>(tmk, tmv, p);
    return check_launch();
}

// fp32 caches with more than four query heads per kv head: the tensor-core step, two
// consumer warps with two of the four stages each (at d = 128 a CTA then fits three to an
// SM; four consumer warps of one stage each measured 7% slower on the 32K-128K-token batch).
#ifndef PKV_F32_TC
#define PKV_F32_TC 1
#endif
#ifndef PKV_F32_TC_NCW
#define PKV_F32_TC_NCW 2
#endif
#ifndef PKV_F32_TC_STAGES
#define PKV_F32_TC_STAGES 4
#endif
constexpr bool kF32Tc = PKV_F32_TC != 0;

template <int D, int GMAX>
int launch_f32_tc(const CUtensorMap &tmk, const CUtensorMap &tmv, const pkv::DecodeParams &p, dim3 grid,
                  cudaStream_t st, bool pdl) {
    using C = pkv::F32TcCfg<D, GMAX, PKV_F32_TC_STAGES, PKV_F32_TC_NCW>;
    static_assert(C::kSmem <= (int)kSmemLimit, "shared memory");
    auto kern = pkv::decode_f32_tc_kernel<D, GMAX, PKV_F32_TC_STAGES, PKV_F32_TC_NCW>;
    static thread_local int configured_device = -1;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    if (configured_device != dev) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem) != cudaSuccess)
            return PKV_ERR_CUDA;
        configured_device = dev;
    }
    if (pdl) return launch_pdl(kern, grid, dim3(C::kThreads), C::kSmem, st, tmk, tmv, p);
    kern<<<grid, C::kThreads, C::kSmem, st>>>(tmk, tmv, p);
    return check_launch();
}

// fp32 caches: the tensor maps of both caches, then the instance for the group size.
template <int D>
int launch_f32(const pkv::DecodeParams &p, dim3 grid, cudaStream_t st, bool pdl) {
    alignas(64) CUtensorMap tmk, tmv;
    int rc;
    if ((rc = encode_cache_map_f32(&tmk, p.k_cache, p.num_blocks, p.num_kv_heads, D)) != PKV_OK) return rc;
    if ((rc = encode_cache_map_f32(&tmv, p.v_cache, p.num_blocks, p.num_kv_heads, D)) != PKV_OK) return rc;
    const int g = p.group;
    if (g == 1) return launch_f32_staged<D, 1>(tmk, tmv, p, grid, st, pdl);
    if (g == 2) return launch_f32_staged<D, 2>(tmk, tmv, p, grid, st, pdl);
    if (g <= 4) return launch_f32_staged<D, 4>(tmk, tmv, p, grid, st, pdl);
    if (kF32Tc) return g <= 8 ? launch_f32_tc<D, 8>(tmk, tmv, p, grid, st, pdl) : launch_f32_tc<D, 16>(tmk, tmv, p, grid, st, pdl);
    if (g <= 8) return launch_f32_staged<D, 8>(tmk, tmv, p, grid, st, pdl);
    return launch_f32_staged<D, 16>(tmk, tmv, p, grid, st, pdl);
}

template <int D, int NT>
int launch_cascade(const CUtensorMap &tmk, const CUtensorMap &tmv, const pkv::DecodeParams &p, dim3 grid,
                   cudaStream_t st) {
    using C = pkv::Bf16Cfg<D, NT, kNstage, kNcw>;
    auto kern = pkv::decode_bf16_cascade_kernel<D, NT, kNstage, kNcw>;
    static thread_local int configured_device = -1;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    if (configured_device != dev) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem) != cudaSuccess)
            return PKV_ERR_CUDA;
        configured_device = dev;
    }
    kern<<<grid, C::kThreads, C::kSmem, st>>>(tmk, tmv, p);
    if (check_launch() != PKV_OK) return PKV_ERR_CUDA;
    const long long rows = (long long)p.num_groups * p.group_size * p.num_q_heads;  // one warp each
    pkv::cascade_reduce_kernel<D>
        <<<(unsigned)((rows + pkv::kReduceWarps - 1) / pkv::kReduceWarps), pkv::kReduceWarps * 32, 0, st>>>(p);
    return check_launch();
}

template <int D>
int launch_reduce(const pkv::DecodeParams &p, pkv_dtype dt, cudaStream_t st) {
    constexpr int PG = 512 / D;  // partition groups: 512 threads per row
    dim3 grid(p.num_q_heads, p.num_seqs);
    const size_t smem = (32 + (size_t)PG * D + (size_t)p.max_parts) * sizeof(float);
    if (dt == PKV_BF16)
        pkv::lse_reduce_kernel<__nv_bfloat16, D, PG><<<grid, D * PG, smem, st>>>(p);
    else
        pkv::lse_reduce_kernel<float, D, PG><<<grid, D * PG, smem, st>>>(p);
    return check_launch();
}


template <int D, bool kUnits>
int launch_prefill_tc(const CUtensorMap &tmq, const CUtensorMap &tmk, const CUtensorMap &tmv,
                      const pkv::PrefillParams &pp, dim3 grid, cudaStream_t st) {
    using C = pkv::TcCfg<D>;
    static_assert(C::kSmem <= (int)kSmemLimit, "shared memory");
    auto kern = kUnits ? pkv::prefill_tc_units_kernel<D> : pkv::prefill_tc_kernel<D>;
    static thread_local int configured_device = -1;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    if (configured_device != dev) {
        // the kernel's register split needs the launch count it was designed for; a build
        // that got fewer registers per thread would wait forever in setmaxnreg.inc
        cudaFuncAttributes fa{};
        if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return PKV_ERR_CUDA;
        if (fa.numRegs * C::kThreads < 128 * C::kLowRegs + C::kTiles * 128 * C::kHighRegs)
            return PKV_ERR_UNSUPPORTED;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem) != cudaSuccess)
            return PKV_ERR_CUDA;
        configured_device = dev;
    }
    kern<<<grid, C::kThreads, C::kSmem, st>>>(tmq, tmk, tmv, pp);
    return check_launch();
}


// Every decode workspace starts with the persistent kernel's arrival counters
// (one per worker, zero between calls); no path writes anything else there,
// so one buffer serves every decode path and shape in turn. Partial softmax
// states follow; each call writes them before it reads them.
constexpr size_t kCounterBytes = PKV_DECODE_COUNTER_BYTES;
static_assert((size_t)kPersistMaxCtas * kPersistWarps * sizeof(int) <= kCounterBytes,
              "one arrival counter per persistent worker");
static_assert(kCounterBytes % 256 == 0, "partials start 256-byte aligned");

size_t grid_workspace_bytes(int num_seqs, int num_q_heads, int head_dim, int max_context_len, int pt) {
    const int mp = max_parts_for(max_context_len, pt);
    if (mp <= 1) return 0;
    return kCounterBytes + (size_t)num_seqs * num_q_heads * mp * (2 + (size_t)head_dim) * sizeof(float);
}

// The counters, then one (max, sum, acc) state per group head for up to two
// cut segments per worker.
size_t persist_workspace_bytes(int num_q_heads, int num_kv_heads, int head_dim) {
    const int g = num_q_heads / num_kv_heads;
    return kCounterBytes + (size_t)kPersistMaxCtas * kPersistWarps * 2 * g * (2 + (size_t)head_dim) * sizeof(float);
}

int sm_count(int *n) {
    static int cached[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    if (dev >= 0 && dev < 64 && cached[dev] > 0) {
        *n = cached[dev];
        return PKV_OK;
    }
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) return PKV_ERR_CUDA;
    if (dev >= 0 && dev < 64) cached[dev] = v;
    *n = v;
    return PKV_OK;
}

template <int D, int NT, int NS, int NW, typename OutT, class WA = pkv::WarpAttn<D, NT>>
int launch_persistent(const CUtensorMap &tmk, const CUtensorMap &tmv, const pkv::DecodeParams &p, cudaStream_t st,
                      bool pdl = false) {
    using C = pkv::PersistCfg<D, NT, NS, NW>;
    static_assert(C::smem_bytes(kPersistMaxSeqs) + 64 <= kSmemLimit, "persistent kernel exceeds shared memory");
    auto kern = pkv::decode_bf16_persistent_kernel<D, NT, NS, NW, OutT, WA>;
    static thread_local int configured_device = -1;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    const size_t max_smem = C::smem_bytes(kPersistMaxSeqs);
    if (configured_device != dev) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)max_smem) != cudaSuccess)
            return PKV_ERR_CUDA;
        configured_device = dev;
    }
    int sms = 0;
    if (sm_count(&sms) != PKV_OK) return PKV_ERR_CUDA;
    const int grid = sms < kPersistMaxCtas ? sms : kPersistMaxCtas;
    if (pdl) return launch_pdl(kern, dim3(grid), dim3(C::kThreads), C::smem_bytes(p.num_seqs), st, tmk, tmv, p);
    kern<<<grid, C::kThreads, C::smem_bytes(p.num_seqs), st>>>(tmk, tmv, p);
    return check_launch();
}

// Head-dim and group-width dispatch of the two bf16 decode kernels: groups
// wider than 8 need two MMA column tiles (the persistent kernel then runs
// half the warps with twice the stages, so their registers fit unspilled).
// One query head per kv head (g = 1) takes the CUDA-core step in both
// kernels: the block's contraction is then a matrix-vector product that
// would fill one of the tensor cores' eight MMA columns.
template <typename OutT, int NS128, int NS64, int NW>
int persistent_by_shape(const CUtensorMap &tmk, const CUtensorMap &tmv, const pkv::DecodeParams &p, cudaStream_t st,
                        bool pdl, int head_dim, int g) {
    if (head_dim == 128) {
        if (g == 1 && kMhaCudaCores)
            return launch_persistent<128, 1, NS128, NW, OutT, pkv::WarpAttnScalar<128>>(tmk, tmv, p, st, pdl);
        return g <= 8 ? launch_persistent<128, 1, NS128, NW, OutT>(tmk, tmv, p, st, pdl)
                      : launch_persistent<128, 2, 2 * NS128, NW / 2, OutT>(tmk, tmv, p, st, pdl);
    }
    if (g == 1 && kMhaCudaCores)
        return launch_persistent<64, 1, NS64, NW, OutT, pkv::WarpAttnScalar<64>>(tmk, tmv, p, st, pdl);
    return g <= 8 ? launch_persistent<64, 1, NS64, NW, OutT>(tmk, tmv, p, st, pdl)
                  : launch_persistent<64, 2, 2 * NS64, NW / 2, OutT>(tmk, tmv, p, st, pdl);
}

template <typename OutT>
int grid_by_shape(const CUtensorMap &tmk, const CUtensorMap &tmv, const pkv::DecodeParams &p, dim3 grid,
                  cudaStream_t st, bool pdl, int head_dim, int g) {
    if (head_dim == 128) {
        if (g == 1 && kMhaCudaCores)
            return launch_bf16<128, 1, OutT, pkv::WarpAttnScalar<128>>(tmk, tmv, p, grid, st, pdl);
        return g <= 8 ? launch_bf16<128, 1, OutT>(tmk, tmv, p, grid, st, pdl)
                      : launch_bf16<128, 2, OutT>(tmk, tmv, p, grid, st, pdl);
    }
    if (g == 1 && kMhaCudaCores)
        return launch_bf16<64, 1, OutT, pkv::WarpAttnScalar<64>>(tmk, tmv, p, grid, st, pdl);
    return g <= 8 ? launch_bf16<64, 1, OutT>(tmk, tmv, p, grid, st, pdl)
                  : launch_bf16<64, 2, OutT>(tmk, tmv, p, grid, st, pdl);
}

// The persistent balanced kernel is chosen for bf16 when asked for
// (PKV_PARTITION_BALANCED), or automatically (partition_tokens == 0) when
// the batch has at least a quarter as many (sequence, kv head) units as the
// GPU has persistent warps; with fewer, longer units the balanced split would
// cut each unit into many segments, and 512-token partitions merged by the
// reduce kernel are faster.
bool use_persistent(pkv_dtype dtype, int partition_tokens, int num_seqs, int num_kv_heads) {
    if (dtype != PKV_BF16 || num_seqs > kPersistMaxSeqs) return false;
    if (partition_tokens == PKV_PARTITION_BALANCED) return true;
    if (partition_tokens != 0) return false;
    int sms = 0;
    if (sm_count(&sms) != PKV_OK) sms = kPersistMaxCtas;
    const int workers = (sms < kPersistMaxCtas ? sms : kPersistMaxCtas) * kPersistWarps;
    return (long long)num_seqs * num_kv_heads * 4 >= workers;
}

// How decode_dispatch ends: launch the attention kernels; launch them right
// after this library's kv_append on the stream (programmatic launch: the
// set-up overlaps the append, cache reads wait for it); or only check.
constexpr int kLaunch = 0, kLaunchAfterAppend = 1, kCheckOnly = 2;

// Shared by the decode entry points once the workspace is known.
int decode_dispatch(void *out, const void *q, const void *k_cache, const void *v_cache, const int32_t *block_tables,
                    const int32_t *context_lens, float scale, int num_kv_heads, int num_seqs, int num_q_heads,
                    int head_dim, int max_blocks_per_seq, int num_blocks, int max_context_len, pkv_dtype dtype,
                    int partition_tokens, void *workspace, size_t workspace_bytes, void *stream, int mode = kLaunch);
}  // namespace

extern "C" {

const char *pkv_status_string(int status) {
    switch (status) {
        case PKV_OK: return "ok";
        case PKV_ERR_ARG: return "bad argument";
        case PKV_ERR_UNSUPPORTED: return "unsupported head_dim, dtype or group size";
        case PKV_ERR_INDEX: return "index out of range";
        case PKV_ERR_OVERLAP: return "copy pairs overlap";
        case PKV_ERR_CUDA: return "CUDA error";
        case PKV_ERR_WORKSPACE: return "workspace missing or too small";
        case PKV_ERR_ALIGN: return "pointer not 16-byte aligned";
        default: return "unknown status";
    }
}

int pkv_version(void) { return kVersion; }

int pkv_decode_partition_tokens(int num_seqs, int num_kv_heads, int max_context_len, int partition_tokens) {
    (void)num_seqs;
    (void)num_kv_heads;
    (void)max_context_len;
    if (partition_tokens > 0) return partition_tokens;
    return kDefaultPartition;  // automatic or balanced: 512 wherever fixed partitions are used
}

size_t pkv_decode_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int max_context_len,
                                  int partition_tokens) {
    if (num_seqs <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0) return 0;
    const int pt = pkv_decode_partition_tokens(num_seqs, num_kv_heads, max_context_len, partition_tokens);
    if (pt <= 0 || pt % 16 != 0) return 0;
    const size_t grid_ws = grid_workspace_bytes(num_seqs, num_q_heads, head_dim, max_context_len, pt);
    if (partition_tokens > 0 || num_q_heads % num_kv_heads != 0) return grid_ws;
    const size_t pers = persist_workspace_bytes(num_q_heads, num_kv_heads, head_dim);
    return pers > grid_ws ? pers : grid_ws;
}

int pkv_decode_persistent(int num_seqs, int num_kv_heads, int partition_tokens, pkv_dtype dtype) {
    if (num_seqs <= 0 || num_kv_heads <= 0 || partition_tokens < PKV_PARTITION_BALANCED) return 0;
    return use_persistent(input_dtype(dtype), partition_tokens, num_seqs, num_kv_heads) ? 1 : 0;
}

int pkv_decode_launches(int num_seqs, int num_kv_heads, int max_context_len, int partition_tokens, pkv_dtype dtype) {
    if (num_seqs <= 0 || num_kv_heads <= 0) return 0;
    if (partition_tokens < PKV_PARTITION_BALANCED) return 0;
    if (use_persistent(input_dtype(dtype), partition_tokens, num_seqs, num_kv_heads)) return 1;
    const int pt = pkv_decode_partition_tokens(num_seqs, 1, max_context_len, partition_tokens);
    if (pt <= 0 || pt % 16 != 0) return 0;
    return max_parts_for(max_context_len, pt) > 1 ? 2 : 1;
}

int paged_decode_attention(void *out, const void *q, const void *k_cache, const void *v_cache,
                           const int32_t *block_tables, const int32_t *context_lens, float scale, int num_kv_heads,
                           int num_seqs, int num_q_heads, int head_dim, int max_blocks_per_seq, int num_blocks,
                           int max_context_len, pkv_dtype dtype, int partition_tokens, void *workspace,
                           size_t workspace_bytes, void *stream) {
    return decode_dispatch(out, q, k_cache, v_cache, block_tables, context_lens, scale, num_kv_heads, num_seqs,
                           num_q_heads, head_dim, max_blocks_per_seq, num_blocks, max_context_len, dtype,
                           partition_tokens, workspace, workspace_bytes, stream);
}

}  // extern "C"

namespace {

int append_impl(const void *k, const void *v, const int64_t *slot_mapping, void *k_cache, void *v_cache,
                int num_tokens, int num_kv_heads, int head_dim, int num_blocks, pkv_dtype dtype, void *stream,
                bool check_only) {
    if (num_tokens < 0 || num_kv_heads <= 0 || num_blocks <= 0) return PKV_ERR_ARG;
    if (!dtype_ok(dtype)) return PKV_ERR_UNSUPPORTED;
    if (head_dim != 64 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
    if (num_tokens == 0) return PKV_OK;
    if (!k || !v || !slot_mapping || !k_cache || !v_cache) return PKV_ERR_ARG;
    if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache)) return PKV_ERR_ALIGN;
    if (check_only) return PKV_OK;
    const int vec_per_row = head_dim * elem_bytes(dtype) / 16;
    const long long total = (long long)num_tokens * num_kv_heads * vec_per_row;
    const int threads = 256;
    const long long blocks = (total + threads - 1) / threads;
    if (blocks > 0x7fffffffLL) return PKV_ERR_UNSUPPORTED;
    pkv::kv_append_kernel<<<(unsigned)blocks, threads, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4 *>(k), static_cast<const uint4 *>(v), slot_mapping, static_cast<uint4 *>(k_cache),
        static_cast<uint4 *>(v_cache), num_tokens, num_kv_heads, vec_per_row, num_blocks);
    return check_launch();
}

}  // namespace

extern "C" {

int kv_append(const void *k, const void *v, const int64_t *slot_mapping, void *k_cache, void *v_cache, int num_tokens,
              int num_kv_heads, int head_dim, int num_blocks, pkv_dtype dtype, void *stream) {
    return append_impl(k, v, slot_mapping, k_cache, v_cache, num_tokens, num_kv_heads, head_dim, num_blocks, dtype,
                       stream, false);
}

int copy_blocks(void *k_cache, void *v_cache, const int64_t *src_dst_pairs, int num_pairs, int num_kv_heads,
                int head_dim, int num_blocks, pkv_dtype dtype, void *stream) {
    return swap_blocks(k_cache, v_cache, num_blocks, k_cache, v_cache, num_blocks, src_dst_pairs, num_pairs,
                       num_kv_heads, head_dim, dtype, stream);
}

}  // extern "C"

namespace {

int move_impl(void *dst_k_cache, void *dst_v_cache, int dst_num_blocks, const void *src_k_cache,
              const void *src_v_cache, int src_num_blocks, const int64_t *src_dst_pairs, int num_pairs,
              int num_kv_heads, int head_dim, pkv_dtype dtype, void *stream, bool check_only) {
    if (num_pairs < 0 || num_kv_heads <= 0 || src_num_blocks <= 0 || dst_num_blocks <= 0) return PKV_ERR_ARG;
    if (!dtype_ok(dtype)) return PKV_ERR_UNSUPPORTED;
    if (head_dim != 64 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
    if (num_pairs == 0) return PKV_OK;
    if (num_pairs > 65535) return PKV_ERR_UNSUPPORTED;
    if (!dst_k_cache || !dst_v_cache || !src_k_cache || !src_v_cache || !src_dst_pairs) return PKV_ERR_ARG;
    if (!aligned16(dst_k_cache) || !aligned16(dst_v_cache) || !aligned16(src_k_cache) || !aligned16(src_v_cache))
        return PKV_ERR_ALIGN;
    if (check_only) return PKV_OK;
    pkv::BlockMove m{};
    m.src[0] = static_cast<const uint4 *>(src_k_cache);
    m.src[1] = static_cast<const uint4 *>(src_v_cache);
    m.dst[0] = static_cast<uint4 *>(dst_k_cache);
    m.dst[1] = static_cast<uint4 *>(dst_v_cache);
    m.src_num_blocks = src_num_blocks;
    m.dst_num_blocks = dst_num_blocks;
    m.vec_per_block = (int64_t)num_kv_heads * 16 * head_dim * elem_bytes(dtype) / 16;
    const int threads = 256;
    int64_t chunks = (m.vec_per_block + threads * 4 - 1) / (threads * 4);
    if (chunks > 1024) chunks = 1024;
    pkv::move_blocks_kernel<<<dim3((unsigned)chunks, num_pairs, 2), threads, 0, static_cast<cudaStream_t>(stream)>>>(
        m, src_dst_pairs);
    return check_launch();
}

}  // namespace

extern "C" {

int swap_blocks(void *dst_k_cache, void *dst_v_cache, int dst_num_blocks, const void *src_k_cache,
                const void *src_v_cache, int src_num_blocks, const int64_t *src_dst_pairs, int num_pairs,
                int num_kv_heads, int head_dim, pkv_dtype dtype, void *stream) {
    return move_impl(dst_k_cache, dst_v_cache, dst_num_blocks, src_k_cache, src_v_cache, src_num_blocks, src_dst_pairs,
                     num_pairs, num_kv_heads, head_dim, dtype, stream, false);
}

int copy_blocks_layers(void *const *k_caches, void *const *v_caches, int num_layers, const int64_t *src_dst_pairs,
                       int num_pairs, int num_kv_heads, int head_dim, int num_blocks, pkv_dtype dtype, void *stream) {
    if (num_pairs < 0 || num_layers < 0 || num_kv_heads <= 0 || num_blocks <= 0) return PKV_ERR_ARG;
    if (!dtype_ok(dtype)) return PKV_ERR_UNSUPPORTED;
    if (head_dim != 64 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
    if (num_pairs == 0 || num_layers == 0) return PKV_OK;
    if (num_pairs > 65535 || num_layers > 32767) return PKV_ERR_UNSUPPORTED;
    if (!k_caches || !v_caches || !src_dst_pairs) return PKV_ERR_ARG;
    pkv::BlockMove m{};
    m.src_k_layers = reinterpret_cast<const uint4 *const *>(k_caches);
    m.src_v_layers = reinterpret_cast<const uint4 *const *>(v_caches);
    m.dst_k_layers = reinterpret_cast<uint4 *const *>(k_caches);
    m.dst_v_layers = reinterpret_cast<uint4 *const *>(v_caches);
    m.src_num_blocks = m.dst_num_blocks = num_blocks;
    m.vec_per_block = (int64_t)num_kv_heads * 16 * head_dim * elem_bytes(dtype) / 16;
    const int threads = 256;
    int64_t chunks = (m.vec_per_block + threads * 4 - 1) / (threads * 4);
    if (chunks > 1024) chunks = 1024;
    pkv::move_blocks_kernel<<<dim3((unsigned)chunks, num_pairs, 2 * num_layers), threads, 0,
                              static_cast<cudaStream_t>(stream)>>>(m, src_dst_pairs);
    return check_launch();
}

int kv_append_layers(const void *const *k, const void *const *v, const int64_t *slot_mapping, void *const *k_caches,
                     void *const *v_caches, int num_layers, int num_tokens, int num_kv_heads, int head_dim,
                     int num_blocks, pkv_dtype dtype, void *stream) {
    if (num_tokens < 0 || num_layers < 0 || num_kv_heads <= 0 || num_blocks <= 0) return PKV_ERR_ARG;
    if (!dtype_ok(dtype)) return PKV_ERR_UNSUPPORTED;
    if (head_dim != 64 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
    if (num_tokens == 0 || num_layers == 0) return PKV_OK;
    if (num_layers > 65535) return PKV_ERR_UNSUPPORTED;
    if (!k || !v || !slot_mapping || !k_caches || !v_caches) return PKV_ERR_ARG;
    const int vec_per_row = head_dim * elem_bytes(dtype) / 16;
    const long long total = (long long)num_tokens * num_kv_heads * vec_per_row;
    const int threads = 256;
    const long long blocks = (total + threads - 1) / threads;
    if (blocks > 0x7fffffffLL) return PKV_ERR_UNSUPPORTED;
    pkv::kv_append_layers_kernel<<<dim3((unsigned)blocks, num_layers), threads, 0,
                                   static_cast<cudaStream_t>(stream)>>>(
        reinterpret_cast<const uint4 *const *>(k), reinterpret_cast<const uint4 *const *>(v), slot_mapping,
        reinterpret_cast<uint4 *const *>(k_caches), reinterpret_cast<uint4 *const *>(v_caches), num_tokens,
        num_kv_heads, vec_per_row, num_blocks);
    return check_launch();
}

int pkv_check_swap_pairs(const int64_t *host_pairs, int num_pairs, int src_num_blocks, int dst_num_blocks) {
    if (num_pairs < 0 || src_num_blocks <= 0 || dst_num_blocks <= 0) return PKV_ERR_ARG;
    if (num_pairs > 0 && !host_pairs) return PKV_ERR_ARG;
    std::unordered_set<int64_t> dsts;
    for (int i = 0; i < num_pairs; ++i) {
        const int64_t s = host_pairs[2 * i], d = host_pairs[2 * i + 1];
        if (s < 0 || s >= src_num_blocks || d < 0 || d >= dst_num_blocks) return PKV_ERR_INDEX;
        if (!dsts.insert(d).second) return PKV_ERR_OVERLAP;
    }
    return PKV_OK;
}

// Partitions of one union unit: at most group_size contexts' blocks.
int cascade_parts(int group_size, int max_context_len, int pt) {
    const long long blocks = (long long)group_size * ((max_context_len + 15) / 16);
    return (int)((blocks * 16 + pt - 1) / pt);
}

size_t pkv_shared_prefix_workspace_bytes(int num_seqs, int num_q_heads, int head_dim, int max_context_len,
                                         int group_size, int partition_tokens) {
    if (num_seqs <= 0 || num_q_heads <= 0 || head_dim <= 0 || max_context_len < 0 || partition_tokens < 0 ||
        group_size <= 0)
        return 0;
    const int pt = pkv_decode_partition_tokens(num_seqs, 1, max_context_len, partition_tokens);
    if (pt % 16 != 0) return 0;
    const int parts = cascade_parts(group_size, max_context_len, pt);
    // the decode counter header (left alone), partition states, then each
    // group's partition count (groups <= sequences)
    return kCounterBytes +
           (size_t)num_seqs * num_q_heads * (size_t)(parts > 0 ? parts : 1) * (2 + (size_t)head_dim) * sizeof(float) +
           (size_t)num_seqs * sizeof(int);
}

int paged_decode_attention_shared_prefix(void *out, const void *q, const void *k_cache, const void *v_cache,
                                         const int32_t *block_tables, const int32_t *context_lens, float scale,
                                         int num_kv_heads, int num_seqs, int num_q_heads, int head_dim,
                                         int max_blocks_per_seq, int num_blocks, int max_context_len,
                                         const int32_t *group_members, const int32_t *shared_blocks, int num_groups,
                                         int group_size, pkv_dtype dtype, int partition_tokens, void *workspace,
                                         size_t workspace_bytes, void *stream) {
    if (num_seqs < 0 || num_kv_heads <= 0 || num_q_heads <= 0 || max_blocks_per_seq <= 0 || num_blocks <= 0 ||
        max_context_len < 0 || partition_tokens < 0 || num_groups < 0 || group_size <= 0)
        return PKV_ERR_ARG;
    if (dtype != PKV_BF16) return PKV_ERR_UNSUPPORTED;
    if (head_dim != 64 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
    if (num_q_heads % num_kv_heads != 0) return PKV_ERR_ARG;
    const int g = num_q_heads / num_kv_heads;
    if (g * group_size > 16 || group_size > 16) return PKV_ERR_UNSUPPORTED;
    if (!std::isfinite(scale)) return PKV_ERR_ARG;
    if (num_seqs > 65535 || num_kv_heads > 65535 || num_groups > 65535) return PKV_ERR_UNSUPPORTED;
    if ((int64_t)num_blocks * num_kv_heads * 16 >= (int64_t(1) << 31)) return PKV_ERR_UNSUPPORTED;
    if (num_seqs == 0) return PKV_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens) return PKV_ERR_ARG;
    if (num_groups > 0 && (!group_members || !shared_blocks)) return PKV_ERR_ARG;
    if (num_groups > num_seqs) return PKV_ERR_ARG;  // every sequence is in exactly one group
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache)) return PKV_ERR_ALIGN;
    const int pt = pkv_decode_partition_tokens(num_seqs, num_kv_heads, max_context_len, partition_tokens);
    if (pt % 16 != 0) return PKV_ERR_ARG;
    const int parts = cascade_parts(group_size, max_context_len, pt);
    if (parts > kMaxParts) return PKV_ERR_UNSUPPORTED;
    const size_t need = pkv_shared_prefix_workspace_bytes(num_seqs, num_q_heads, head_dim, max_context_len,
                                                          group_size, partition_tokens);
    if (!workspace || workspace_bytes < need || !aligned16(workspace)) return PKV_ERR_WORKSPACE;

    pkv::DecodeParams p{};
    p.out = out;
    p.q = q;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.scale_log2 = (float)((double)scale * 1.4426950408889634);
    p.num_seqs = num_seqs;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = num_kv_heads;
    p.group = g;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.num_blocks = num_blocks;
    p.max_context_len = max_context_len;
    p.part_blocks = pt / 16;
    p.max_parts = parts > 0 ? parts : 1;
    p.pre_parts = 0;
    p.ws_ml = reinterpret_cast<float *>(static_cast<char *>(workspace) + kCounterBytes);
    p.ws_o = p.ws_ml + (size_t)num_seqs * num_q_heads * p.max_parts * 2;
    p.counters = reinterpret_cast<int *>(p.ws_o + (size_t)num_seqs * num_q_heads * p.max_parts * head_dim);
    p.group_members = group_members;
    p.shared_blocks = shared_blocks;
    p.num_groups = num_groups;
    p.group_size = group_size;
    alignas(64) CUtensorMap tmk, tmv;
    int rc;
    if ((rc = encode_cache_map(&tmk, k_cache, num_blocks, num_kv_heads, head_dim)) != PKV_OK) return rc;
    if ((rc = encode_cache_map(&tmv, v_cache, num_blocks, num_kv_heads, head_dim)) != PKV_OK) return rc;
    if (num_groups == 0) return PKV_OK;
    const dim3 grid(p.max_parts, num_kv_heads, num_groups);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool wide = g * group_size > 8;
    if (head_dim == 128)
        return wide ? launch_cascade<128, 2>(tmk, tmv, p, grid, st) : launch_cascade<128, 1>(tmk, tmv, p, grid, st);
    return wide ? launch_cascade<64, 2>(tmk, tmv, p, grid, st) : launch_cascade<64, 1>(tmk, tmv, p, grid, st);
}

int paged_prefill_attention(void *out, const void *q, const void *k_cache, const void *v_cache,
                            const int32_t *block_tables, const int32_t *context_lens, const int32_t *query_start,
                            float scale, int num_kv_heads, int num_seqs, int num_q_heads, int head_dim,
                            int max_blocks_per_seq, int num_blocks, int num_queries, int max_query_len,
                            int max_context_len, pkv_dtype dtype, void *stream) {
    if (num_seqs < 0 || num_kv_heads <= 0 || num_q_heads <= 0 || max_blocks_per_seq <= 0 || num_blocks <= 0 ||
        max_context_len < 0 || max_query_len < 0 || num_queries < 0)
        return PKV_ERR_ARG;
    if (dtype != PKV_BF16) return PKV_ERR_UNSUPPORTED;
    if (head_dim != 64 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
    if (num_q_heads % num_kv_heads != 0) return PKV_ERR_ARG;
    const int g = num_q_heads / num_kv_heads;
    if (g > 64) return PKV_ERR_UNSUPPORTED;
    if (!std::isfinite(scale)) return PKV_ERR_ARG;
    if (num_seqs > 65535 || num_kv_heads > 65535) return PKV_ERR_UNSUPPORTED;
    if ((int64_t)num_blocks * num_kv_heads * 16 >= (int64_t(1) << 31)) return PKV_ERR_UNSUPPORTED;
    const int tile_tokens = 128 / g;  // 128 query rows per tile, two tiles per CTA
    const int tiles = (max_query_len + tile_tokens - 1) / tile_tokens;
    const int pairs = (tiles + 1) / 2;
    if (pairs > 65535) return PKV_ERR_UNSUPPORTED;
    if (num_seqs == 0 || max_query_len == 0 || num_queries == 0) return PKV_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens || !query_start) return PKV_ERR_ARG;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache)) return PKV_ERR_ALIGN;

    pkv::PrefillParams pp{};
    pkv::DecodeParams &p = pp.d;
    p.out = out;
    p.q = q;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.scale_log2 = (float)((double)scale * 1.4426950408889634);
    p.num_seqs = num_seqs;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = num_kv_heads;
    p.group = g;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.num_blocks = num_blocks;
    p.max_context_len = max_context_len;
    pp.query_start = query_start;
    pp.tile_tokens = tile_tokens;
    pp.max_query_len = max_query_len;
    pp.num_queries = num_queries;
    alignas(64) CUtensorMap tmk, tmv;
    int rc;
    // CTA order. Whole prompts (context not much longer than the new tokens):
    // the pair index slowest, so every sequence's last (longest) pair starts
    // before any shorter one. Chunks after a cached context at least as long
    // as the chunk: one sequence at a time (longest first), so the pairs of a
    // (sequence, kv head) read its K/V from L2 -- there each pair attends the
    // whole cached context, and re-reading it from DRAM dominates.
    pp.seq_major = max_context_len >= 2 * max_query_len ? 1 : 0;
    // Many (sequence, kv head) units of whole prompts: one CTA per unit takes all its pairs, so
    // each CTA's set-up is paid once and the next pair's loads overlap the current pair's end.
    int sms = 0;
    if (sm_count(&sms) != PKV_OK) return PKV_ERR_CUDA;
    const bool units = kPrefillUnits && !pp.seq_major && (long long)num_seqs * num_kv_heads >= 4LL * sms;
    const dim3 grid = units          ? dim3(num_kv_heads, num_seqs)
                      : pp.seq_major ? dim3(num_kv_heads, pairs, num_seqs)
                                     : dim3(num_kv_heads, num_seqs, pairs);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    alignas(64) CUtensorMap tmq;
    if ((rc = encode_q_map(&tmq, q, num_queries, num_q_heads, head_dim, g, tile_tokens)) != PKV_OK) return rc;
    if ((rc = encode_cache_map(&tmk, k_cache, num_blocks, num_kv_heads, head_dim, true)) != PKV_OK) return rc;
    if ((rc = encode_cache_map(&tmv, v_cache, num_blocks, num_kv_heads, head_dim, true)) != PKV_OK) return rc;
    if (units)
        return head_dim == 128 ? launch_prefill_tc<128, true>(tmq, tmk, tmv, pp, grid, st)
                               : launch_prefill_tc<64, true>(tmq, tmk, tmv, pp, grid, st);
    return head_dim == 128 ? launch_prefill_tc<128, false>(tmq, tmk, tmv, pp, grid, st)
                           : launch_prefill_tc<64, false>(tmq, tmk, tmv, pp, grid, st);
}

int pkv_check_copy_pairs(const int64_t *host_pairs, int num_pairs, int num_blocks) {
    if (num_pairs < 0 || num_blocks <= 0) return PKV_ERR_ARG;
    if (num_pairs > 0 && !host_pairs) return PKV_ERR_ARG;
    std::unordered_set<int64_t> srcs, dsts;
    for (int i = 0; i < num_pairs; ++i) {
        const int64_t s = host_pairs[2 * i], d = host_pairs[2 * i + 1];
        if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks) return PKV_ERR_INDEX;
        srcs.insert(s);
        if (!dsts.insert(d).second) return PKV_ERR_OVERLAP;
    }
    for (int64_t d : dsts)
        if (srcs.count(d)) return PKV_ERR_OVERLAP;
    return PKV_OK;
}

int pkv_validate(const int32_t *block_tables, const int32_t *context_lens, int num_seqs, int max_blocks_per_seq,
                 int num_blocks, int max_context_len, int32_t *dev_err_word, void *stream) {
    if (num_seqs < 0 || max_blocks_per_seq <= 0 || num_blocks <= 0 || max_context_len < 0 || !dev_err_word)
        return PKV_ERR_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(dev_err_word, 0, sizeof(int32_t), st) != cudaSuccess) return PKV_ERR_CUDA;
    if (num_seqs == 0) return PKV_OK;
    if (!block_tables || !context_lens) return PKV_ERR_ARG;
    pkv::validate_tables_kernel<<<num_seqs, 128, 0, st>>>(block_tables, context_lens, max_blocks_per_seq, num_blocks,
                                                          max_context_len, dev_err_word);
    return check_launch();
}

int pkv_validate_slots(const int64_t *slot_mapping, int num_tokens, int num_blocks, int32_t *dev_err_word,
                       void *stream) {
    if (num_tokens < 0 || num_blocks <= 0 || !dev_err_word) return PKV_ERR_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(dev_err_word, 0, sizeof(int32_t), st) != cudaSuccess) return PKV_ERR_CUDA;
    if (num_tokens == 0) return PKV_OK;
    if (!slot_mapping) return PKV_ERR_ARG;
    pkv::validate_slots_kernel<<<(num_tokens + 255) / 256, 256, 0, st>>>(slot_mapping, num_tokens, num_blocks,
                                                                        dev_err_word);
    return check_launch();
}

int pkv_device_error(uint32_t *value, int clear) {
    if (!value) return PKV_ERR_ARG;
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, pkv::g_dev_error, sizeof(v)) != cudaSuccess) return PKV_ERR_CUDA;
    *value = v;
    if (clear) {
        const unsigned int zero = 0;
        if (cudaMemcpyToSymbol(pkv::g_dev_error, &zero, sizeof(zero)) != cudaSuccess) return PKV_ERR_CUDA;
    }
    return PKV_OK;
}

}  // extern "C"


namespace {

int decode_dispatch(void *out, const void *q, const void *k_cache, const void *v_cache, const int32_t *block_tables,
                    const int32_t *context_lens, float scale, int num_kv_heads, int num_seqs, int num_q_heads,
                    int head_dim, int max_blocks_per_seq, int num_blocks, int max_context_len, pkv_dtype dtype,
                    int partition_tokens, void *workspace, size_t workspace_bytes, void *stream, int mode) {
    if (num_seqs < 0 || num_kv_heads <= 0 || num_q_heads <= 0 || max_blocks_per_seq <= 0 || num_blocks <= 0 ||
        max_context_len < 0 || partition_tokens < PKV_PARTITION_BALANCED)
        return PKV_ERR_ARG;
    if (!dtype_ok(input_dtype(dtype))) return PKV_ERR_UNSUPPORTED;
    const bool f32_out = dtype == PKV_BF16_OUT_F32;
    dtype = input_dtype(dtype);
    if (head_dim != 64 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
    if (num_q_heads % num_kv_heads != 0) return PKV_ERR_ARG;
    const int g = num_q_heads / num_kv_heads;
    if (g > 16) return PKV_ERR_UNSUPPORTED;
    if (!std::isfinite(scale)) return PKV_ERR_ARG;
    if (num_seqs > 65535 || num_kv_heads > 65535) return PKV_ERR_UNSUPPORTED;
    if ((int64_t)num_blocks * num_kv_heads * 16 >= (int64_t(1) << 31)) return PKV_ERR_UNSUPPORTED;
    if (num_seqs == 0) return PKV_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens) return PKV_ERR_ARG;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache)) return PKV_ERR_ALIGN;
    const int pt = pkv_decode_partition_tokens(num_seqs, num_kv_heads, max_context_len, partition_tokens);
    if (pt % 16 != 0) return PKV_ERR_ARG;
    const int mp = max_parts_for(max_context_len, pt);
    const bool persistent = use_persistent(dtype, partition_tokens, num_seqs, num_kv_heads);
    if (!persistent && mp > kMaxParts) return PKV_ERR_UNSUPPORTED;
    const size_t need = pkv_decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim, max_context_len,
                                                   partition_tokens);
    if (need > 0 && (!workspace || workspace_bytes < need || !aligned16(workspace))) return PKV_ERR_WORKSPACE;
    if (mode == kCheckOnly) return PKV_OK;
    const bool pdl = mode == kLaunchAfterAppend;

    pkv::DecodeParams p{};
    p.out = out;
    p.q = q;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.scale_log2 = (float)((double)scale * 1.4426950408889634);
    p.num_seqs = num_seqs;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = num_kv_heads;
    p.group = g;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.num_blocks = num_blocks;
    p.max_context_len = max_context_len;
    p.part_blocks = pt / 16;
    p.max_parts = mp;
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    if (persistent) {
        p.counters = static_cast<int *>(workspace);
        p.partials = reinterpret_cast<float *>(static_cast<char *>(workspace) + kCounterBytes);
        alignas(64) CUtensorMap tmk, tmv;
        int rc;
        if ((rc = encode_cache_map(&tmk, k_cache, num_blocks, num_kv_heads, head_dim)) != PKV_OK) return rc;
        if ((rc = encode_cache_map(&tmv, v_cache, num_blocks, num_kv_heads, head_dim)) != PKV_OK) return rc;
        constexpr int ns128 = PKV_PERSIST_STAGES_D128, ns64 = PKV_PERSIST_STAGES_D64, nw = kPersistWarps;
        return f32_out ? persistent_by_shape<float, ns128, ns64, nw>(tmk, tmv, p, st, pdl, head_dim, g)
                       : persistent_by_shape<__nv_bfloat16, ns128, ns64, nw>(tmk, tmv, p, st, pdl, head_dim, g);
    }

    const size_t grid_ws = grid_workspace_bytes(num_seqs, num_q_heads, head_dim, max_context_len, pt);
    p.ws_ml = grid_ws ? reinterpret_cast<float *>(static_cast<char *>(workspace) + kCounterBytes) : nullptr;
    p.ws_o = grid_ws ? p.ws_ml + (size_t)num_seqs * num_q_heads * mp * 2 : nullptr;
    dim3 grid(mp, num_kv_heads, num_seqs);
    int rc;
    if (dtype == PKV_BF16) {
        alignas(64) CUtensorMap tmk, tmv;
        if ((rc = encode_cache_map(&tmk, k_cache, num_blocks, num_kv_heads, head_dim)) != PKV_OK) return rc;
        if ((rc = encode_cache_map(&tmv, v_cache, num_blocks, num_kv_heads, head_dim)) != PKV_OK) return rc;
        rc = f32_out ? grid_by_shape<float>(tmk, tmv, p, grid, st, pdl, head_dim, g)
                     : grid_by_shape<__nv_bfloat16>(tmk, tmv, p, grid, st, pdl, head_dim, g);
    } else {
        rc = head_dim == 128 ? launch_f32<128>(p, grid, st, pdl) : launch_f32<64>(p, grid, st, pdl);
    }
    if (rc != PKV_OK) return rc;
    const pkv_dtype out_dt = f32_out ? PKV_F32 : dtype;
    if (mp > 1) rc = head_dim == 128 ? launch_reduce<128>(p, out_dt, st) : launch_reduce<64>(p, out_dt, st);
    return rc;
}

}  // namespace

// ---------------------------------------------------------------------------
// Decode without a caller-provided workspace (see pagedkv.h): the scratch is a
// file-scope device array whose device address is looked up once per device.
// ---------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_static_workspace[PKV_STATIC_WORKSPACE_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_static_workspace_mu;
void *g_static_workspace_ptr[kMaxDevices] = {};

// Device address of g_static_workspace on the current device. In host code the
// array's name is only a host-side stand-in, so it is resolved with
// cudaGetSymbolAddress, with that device current, the first time.
int static_workspace_address(void **ptr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return PKV_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_static_workspace_mu);
    if (!g_static_workspace_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess || !p) return PKV_ERR_CUDA;
        g_static_workspace_ptr[dev] = p;
    }
    *ptr = g_static_workspace_ptr[dev];
    return PKV_OK;
}

}  // namespace

extern "C" int paged_decode_attention_static_workspace(void *out, const void *q, const void *k_cache,
                                                       const void *v_cache, const int32_t *block_tables,
                                                       const int32_t *context_lens, float scale, int num_kv_heads,
                                                       int num_seqs, int num_q_heads, int head_dim,
                                                       int max_blocks_per_seq, int num_blocks, int max_context_len,
                                                       pkv_dtype dtype, int partition_tokens, void *stream) {
    if (num_seqs < 0 || num_kv_heads <= 0 || num_q_heads <= 0 || head_dim <= 0 || max_context_len < 0 ||
        partition_tokens < PKV_PARTITION_BALANCED)
        return PKV_ERR_ARG;
    const size_t need = pkv_decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim, max_context_len,
                                                   partition_tokens);
    if (need > PKV_STATIC_WORKSPACE_BYTES) return PKV_ERR_WORKSPACE;
    void *workspace = nullptr;
    if (need > 0 && num_seqs > 0) {
        const int rc = static_workspace_address(&workspace);
        if (rc != PKV_OK) return rc;
    }
    return decode_dispatch(out, q, k_cache, v_cache, block_tables, context_lens, scale, num_kv_heads, num_seqs,
                           num_q_heads, head_dim, max_blocks_per_seq, num_blocks, max_context_len, dtype,
                           partition_tokens, workspace, workspace ? (size_t)PKV_STATIC_WORKSPACE_BYTES : 0, stream);
}

// ---------------------------------------------------------------------------
// One decode step in one call (see pagedkv.h): copy-on-write copies, the KV
// append, then attention. The library launches the append itself, so it knows
// the kernel right before the attention writes only the caches: the attention
// is launched programmatically and reads tables, lengths and queries while the
// append runs, waiting for it only before its first cache read.
// ---------------------------------------------------------------------------
extern "C" int paged_decode_step(void *out, const void *q, void *k_cache, void *v_cache, const int32_t *block_tables,
                                 const int32_t *context_lens, float scale, int num_kv_heads, int num_seqs,
                                 int num_q_heads, int head_dim, int max_blocks_per_seq, int num_blocks,
                                 int max_context_len, pkv_dtype dtype, int partition_tokens, void *workspace,
                                 size_t workspace_bytes, const void *k_new, const void *v_new,
                                 const int64_t *slot_mapping, int num_tokens, const int64_t *src_dst_pairs,
                                 int num_pairs, void *stream) {
    int rc;
    const pkv_dtype cache_dt = input_dtype(dtype);  // what append and copy move
    // every argument is checked before anything is launched
    if ((rc = decode_dispatch(out, q, k_cache, v_cache, block_tables, context_lens, scale, num_kv_heads, num_seqs,
                              num_q_heads, head_dim, max_blocks_per_seq, num_blocks, max_context_len, dtype,
                              partition_tokens, workspace, workspace_bytes, stream, kCheckOnly)) != PKV_OK)
        return rc;
    if ((rc = append_impl(k_new, v_new, slot_mapping, k_cache, v_cache, num_tokens, num_kv_heads, head_dim, num_blocks,
                          cache_dt, stream, true)) != PKV_OK)
        return rc;
    if ((rc = move_impl(k_cache, v_cache, num_blocks, k_cache, v_cache, num_blocks, src_dst_pairs, num_pairs,
                        num_kv_heads, head_dim, cache_dt, stream, true)) != PKV_OK)
        return rc;
    if ((rc = move_impl(k_cache, v_cache, num_blocks, k_cache, v_cache, num_blocks, src_dst_pairs, num_pairs,
                        num_kv_heads, head_dim, cache_dt, stream, false)) != PKV_OK)
        return rc;
    if ((rc = append_impl(k_new, v_new, slot_mapping, k_cache, v_cache, num_tokens, num_kv_heads, head_dim, num_blocks,
                          cache_dt, stream, false)) != PKV_OK)
        return rc;
    return decode_dispatch(out, q, k_cache, v_cache, block_tables, context_lens, scale, num_kv_heads, num_seqs,
                           num_q_heads, head_dim, max_blocks_per_seq, num_blocks, max_context_len, dtype,
                           partition_tokens, workspace, workspace_bytes, stream,
                           num_tokens > 0 ? kLaunchAfterAppend : kLaunch);
}
