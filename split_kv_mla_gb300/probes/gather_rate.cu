// gather_rate.cu -- how fast can one CTA per SM stream random 576-byte pool rows
// into shared memory, with nothing else to do?
//
// The split kernel's fetch: 128-row blocks of fused fp8 rows (512 latent + 64
// RoPE bytes) at random slots of a page-size-1 pool, two blocks in flight per
// CTA, each block in the 128-byte-swizzled layout the tensor cores read.  This
// program runs that fetch alone, by four mechanisms:
//
//   tma_gather4   TMA tile::gather4: per four rows, four 128-byte latent boxes
//                 and one 64-byte RoPE box (the split kernel's copies)
//   tma+cp_async  the four latent boxes by TMA, the RoPE bytes by 16-byte cp.async
//   cp_async16    every 16-byte chunk by cp.async into the same layout
//   bulk_row      one 576-byte cp.async.bulk per row, row-major (a layout the
//                 tensor cores cannot read; shown as the copy engine's ceiling)
//
// Slots are a seeded permutation of a 1 Mi-row pool (604 MB), and successive
// launches read disjoint slot sets, so the rows come from DRAM.  Each
// configuration is timed over 20 back-to-back launches (CUDA events), median of
// three.  Output: one CSV line per configuration with microseconds per launch,
// GB/s of rows delivered, and the mean SM cycles warp 0 spent issuing one block.
//
// Every wait is bounded; a timeout sets an error word that the host reports.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <random>
#include <vector>

#include "../csrc/mla_sm100.cuh"

using namespace mla::sm100;

namespace {

constexpr int kRowBytes = 576;
constexpr int kBlockN = 128;
constexpr int kStageBytes = kBlockN * kRowBytes;   // 73,728
constexpr int kLatChunk = kBlockN * 128;           // one 128-byte column chunk of a block
constexpr int kStages = 2;
constexpr int kMaxBlocks = 16;
constexpr int kThreads = 512;
constexpr long long kRows = 1 << 20;

enum Mode { kTmaGather4 = 0, kTmaCpAsync = 1, kCpAsync16 = 2, kBulkRow = 3 };
const char* kModeName[] = {"tma_gather4", "tma+cp_async", "cp_async16", "bulk_row"};

struct Args {
    const uint8_t* pool;
    const int* slots;   // kRows entries
    long long slot_off;
    int nblk, warps, mode;
    long long* issue_cycles;   // per CTA: warp 0's mean cycles issuing a block
    int* err;
};

__device__ __forceinline__ void cp_async16(uint8_t* dst, const uint8_t* src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
                 : "memory");
}

__device__ __forceinline__ void cp_async_arrive(uint64_t* bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void bulk_copy(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes),
          "r"(smem_u32(bar))
        : "memory");
}

// Destination of 16-byte chunk c (0..35) of block row r in the swizzled stage:
// latent chunks in four 128-byte column chunks (128-byte swizzle), RoPE chunks in
// the 64-byte-swizzled fifth.
__device__ __forceinline__ uint8_t* chunk_dst(uint8_t* stage, int r, int c)
{
    if (c < 32) return stage + (c >> 3) * kLatChunk + r * 128 + (((c & 7) ^ (r & 7)) << 4);
    return stage + 4 * kLatChunk + r * 64 + ((((c - 32) ^ ((r >> 1) & 3))) << 4);
}

__global__ void __launch_bounds__(kThreads, 1)
gather_rate_kernel(const __grid_constant__ CUtensorMap tm_lat,
                   const __grid_constant__ CUtensorMap tm_rope, const Args a)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    int* slots = reinterpret_cast<int*>(smem + kStages * kStageBytes);
    uint64_t* full = reinterpret_cast<uint64_t*>(slots + kMaxBlocks * kBlockN);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(full + kStages);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int T = a.warps * 32;
    if (smem_u32(smem) & 1023u) {
        if (tid == 0) atomicOr(a.err, 4);
        return;
    }
    if (tid == 0) {
        // arrivals per phase: one per issuing warp (TMA / bulk), plus one per
        // thread for the cp.async completions
        const int count = a.mode == kTmaGather4 || a.mode == kBulkRow ? a.warps
                          : a.mode == kTmaCpAsync                     ? a.warps + T
                                                                      : T;
        for (int i = 0; i < kStages; ++i) mbar_init(&full[i], count);
        *abort_flag = 0;
        fence_mbar_init();
    }
    const int* g = a.slots + a.slot_off + (long long)blockIdx.x * a.nblk * kBlockN;
    for (int i = tid; i < a.nblk * kBlockN; i += kThreads) slots[i] = g[i];
    __syncthreads();
    if (warp >= a.warps) return;

    long long cycles = 0;
    int j = 0;
    for (; j < a.nblk; ++j) {
        const int st = j % kStages;
        if (j >= kStages &&
            !mbar_wait_or_abort(&full[st], ((j / kStages) - 1) & 1, abort_flag)) {
            if (lane == 0) atomicOr(a.err, 1);
            break;
        }
        uint8_t* stage = smem + st * kStageBytes;
        const int* bs = slots + j * kBlockN;
        const long long t0 = clock64();
        if (a.mode == kTmaGather4 || a.mode == kTmaCpAsync) {
            const int boxes = a.mode == kTmaGather4 ? 5 : 4;
            const int items = 32 * boxes;
            const int per = (items + a.warps - 1) / a.warps;
            const int i0 = min(items, warp * per), i1 = min(items, i0 + per);
            uint32_t bytes = 0;
            for (int i = i0; i < i1; ++i) bytes += (i % boxes) < 4 ? 512u : 256u;
            if (lane == 0) mbar_arrive_expect_tx(&full[st], bytes);
            __syncwarp();
            for (int i = i0 + lane; i < i1; i += 32) {
                const int grp = i / boxes, box = i % boxes;
                uint8_t* dst = box < 4 ? stage + box * kLatChunk + grp * 512
                                       : stage + 4 * kLatChunk + grp * 256;
                tma_gather4(dst, box < 4 ? (const void*)&tm_lat : (const void*)&tm_rope,
                            box < 4 ? box * 128 : 512, bs[4 * grp], bs[4 * grp + 1],
                            bs[4 * grp + 2], bs[4 * grp + 3], &full[st]);
            }
            if (a.mode == kTmaCpAsync) {
                for (int i = tid; i < kBlockN * 4; i += T) {
                    const int r = i >> 2, c = 32 + (i & 3);
                    cp_async16(chunk_dst(stage, r, c),
                               a.pool + (long long)bs[r] * kRowBytes + c * 16);
                }
                cp_async_arrive(&full[st]);
            }
        } else if (a.mode == kCpAsync16) {
            for (int i = tid; i < kBlockN * 36; i += T) {
                const int r = i / 36, c = i % 36;
                cp_async16(chunk_dst(stage, r, c), a.pool + (long long)bs[r] * kRowBytes + c * 16);
            }
            cp_async_arrive(&full[st]);
        } else {
            const int per = (kBlockN + a.warps - 1) / a.warps;
            const int r0 = min(kBlockN, warp * per), r1 = min(kBlockN, r0 + per);
            if (lane == 0) mbar_arrive_expect_tx(&full[st], (uint32_t)(r1 - r0) * kRowBytes);
            __syncwarp();
            for (int r = r0 + lane; r < r1; r += 32)
                bulk_copy(stage + r * kRowBytes, a.pool + (long long)bs[r] * kRowBytes,
                          kRowBytes, &full[st]);
        }
        cycles += clock64() - t0;
    }
    // the blocks still in flight land before the CTA exits
    volatile int drain_abort = 0;
    for (int k = max(0, j - kStages); k < j; ++k)
        if (!mbar_wait_or_abort(&full[k % kStages], (k / kStages) & 1, &drain_abort) && lane == 0)
            atomicOr(a.err, 2);
    asm volatile("cp.async.wait_all;" ::: "memory");
    if (tid == 0) a.issue_cycles[blockIdx.x] = cycles / max(1, a.nblk);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
}

// One-row boxes of `box` bytes over the pool (the shape tile::gather4 reads).
bool row_map(CUtensorMap* m, const void* pool, int box, CUtensorMapSwizzle sw)
{
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t gdim[2] = {(cuuint64_t)kRowBytes, (cuuint64_t)kRows};
    cuuint64_t gstr[1] = {(cuuint64_t)kRowBytes};
    cuuint32_t bdim[2] = {(cuuint32_t)box, 1};
    cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(pool), gdim, gstr, bdim, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

#define CHECK(x)                                                                          \
    do {                                                                                  \
        cudaError_t e_ = (x);                                                             \
        if (e_ != cudaSuccess) {                                                          \
            std::printf("CUDA error %s at line %d\n", cudaGetErrorString(e_), __LINE__);  \
            return 1;                                                                     \
        }                                                                                 \
    } while (0)

int main()
{
    uint8_t* pool = nullptr;
    CHECK(cudaMalloc(&pool, (size_t)kRows * kRowBytes));
    CHECK(cudaMemset(pool, 0x31, (size_t)kRows * kRowBytes));
    std::vector<int> perm(kRows);
    for (long long i = 0; i < kRows; ++i) perm[i] = (int)i;
    std::mt19937 rng(7);
    std::shuffle(perm.begin(), perm.end(), rng);
    int* slots = nullptr;
    CHECK(cudaMalloc(&slots, kRows * sizeof(int)));
    CHECK(cudaMemcpy(slots, perm.data(), kRows * sizeof(int), cudaMemcpyHostToDevice));
    long long* cycles = nullptr;
    int* err = nullptr;
    CHECK(cudaMalloc(&cycles, 1024 * sizeof(long long)));
    CHECK(cudaMalloc(&err, sizeof(int)));
    CHECK(cudaMemset(err, 0, sizeof(int)));
    CUtensorMap tm_lat, tm_rope;
    if (!row_map(&tm_lat, pool, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !row_map(&tm_rope, pool, 64, CU_TENSOR_MAP_SWIZZLE_64B)) {
        std::printf("tensor map encode failed\n");
        return 1;
    }
    const int smem = kStages * kStageBytes + kMaxBlocks * kBlockN * 4 + 64;
    CHECK(cudaFuncSetAttribute(gather_rate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               smem));
    int sms = 0;
    CHECK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0));
    cudaEvent_t e0, e1;
    CHECK(cudaEventCreate(&e0));
    CHECK(cudaEventCreate(&e1));
    constexpr int kLaunches = 20;
    std::printf("mode,ctas,blocks_per_cta,issuing_warps,us_per_launch,GBps,issue_cycles_per_block\n");
    for (int nblk : {4, 16})
        for (int ctas : {128, sms})
            for (int mode = 0; mode < 4; ++mode)
                for (int warps : {7, 16}) {
                    if (ctas > 1024) continue;
                    const long long per_launch = (long long)ctas * nblk * kBlockN;
                    const int sets = (int)(kRows / per_launch);   // disjoint slot sets
                    Args a{pool, slots, 0, nblk, warps, mode, cycles, err};
                    std::vector<float> t;
                    for (int rep = 0; rep < 4; ++rep) {
                        CHECK(cudaEventRecord(e0));
                        for (int l = 0; l < kLaunches; ++l) {
                            a.slot_off = (long long)((rep * kLaunches + l) % sets) * per_launch;
                            gather_rate_kernel<<<ctas, kThreads, smem>>>(tm_lat, tm_rope, a);
                        }
                        CHECK(cudaGetLastError());
                        CHECK(cudaEventRecord(e1));
                        CHECK(cudaEventSynchronize(e1));
                        float ms = 0.f;
                        CHECK(cudaEventElapsedTime(&ms, e0, e1));
                        if (rep > 0) t.push_back(ms * 1e3f / kLaunches);
                    }
                    int herr = 0;
                    CHECK(cudaMemcpy(&herr, err, sizeof(int), cudaMemcpyDeviceToHost));
                    if (herr) {
                        std::printf("device error word %d (mode %s)\n", herr, kModeName[mode]);
                        return 2;
                    }
                    std::vector<long long> c(ctas);
                    CHECK(cudaMemcpy(c.data(), cycles, ctas * sizeof(long long),
                                     cudaMemcpyDeviceToHost));
                    double mc = 0.0;
                    for (long long v : c) mc += (double)v / ctas;
                    std::sort(t.begin(), t.end());
                    const double us = t[t.size() / 2];
                    std::printf("%s,%d,%d,%d,%.2f,%.0f,%.0f\n", kModeName[mode], ctas, nblk, warps,
                                us, (double)per_launch * kRowBytes / (us * 1e3), mc);
                }
    return 0;
}
