// memory_probe.cu -- standalone measurements of the memory-system floors the
// decode attention kernels run against (not part of the library):
//   stream   152 (or 76) CTAs stream a K and a V tensor [n_kv][256] f16
//            through a ring of 32 KiB shared-memory stages filled by 2-D TMA
//            boxes of 64 dims x 128 rows (the attention kernels' pattern),
//            with no compute: the consumer frees each stage as it lands.
//   l2       the same, every CTA reading the same 8 MiB (L2-resident).
//   fresh    152 CTAs each write an 8 KiB block, pass a grid barrier, then
//            one warp per CTA reads one 128-byte line of 20 other CTAs'
//            blocks (independent loads) and times them; then 20 more lines
//            of the same blocks (the lines are warm).
//   dsmem    clusters of 2 or 8 CTAs: every CTA pushes 96 KiB into the shared
//            memory of the next CTA of its cluster with 16-byte
//            st.shared::cluster stores (all 256 threads), then a cluster
//            barrier; the push time per CTA gives GB/s per SM.
// Every wait is bounded (0.2 s); a wait that gives up sets a status bit that
// the host prints. Build and run: python -m gqa_kv_head_gb300.probes
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <cstring>

#include "fr_sm100.cuh"

using namespace fr::sm100;

constexpr int kHd = 256;
constexpr uint64_t kLimitNs = 200000000ull;

template <int R>
__global__ void __launch_bounds__(64, 1) stream_kernel(const __grid_constant__ CUtensorMap k,
                                                      const __grid_constant__ CUtensorMap v, int keys_per_cta,
                                                      int same_region, unsigned* status) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + R * 32768);
    const int tid = threadIdx.x;
    const int k0 = same_region ? 0 : blockIdx.x * keys_per_cta;
    const int n_pieces = (keys_per_cta / 128) * 4;          // per 128-key tile: K dims 0-127, 128-255, then V
    if (tid == 0) {
        for (int s = 0; s < R; ++s) {
            mbar_init(smem_addr(&bars[s]), 1);
            mbar_init(smem_addr(&bars[R + s]), 1);
        }
        mbar_fence_init();
    }
    __syncthreads();
    int issued = 0;
    if (tid == 0) {
        for (int p = 0; p < n_pieces; ++p) {
            const int st = p % R;
            if (p >= R && !mbar_wait(smem_addr(&bars[R + st]), ((p / R) - 1) & 1, kLimitNs)) {
                atomicOr(status, 1u);
                break;
            }
            const uint32_t dst = smem_addr(sm + st * 32768);
            const uint32_t fb = smem_addr(&bars[st]);
            const int tile = p / 4, q = p % 4;
            const CUtensorMap* m = q < 2 ? &k : &v;
            mbar_expect_tx(fb, 32768u);
            tma_load_2d(dst, m, (q & 1) * 128, k0 + tile * 128, fb);
            tma_load_2d(dst + 16384, m, (q & 1) * 128 + 64, k0 + tile * 128, fb);
            issued = p + 1;
        }
        // drain: every issued copy has landed before the CTA exits
        for (int p = issued > R ? issued - R : 0; p < issued; ++p)
            if (!mbar_wait(smem_addr(&bars[p % R]), (p / R) & 1, kLimitNs)) atomicOr(status, 4u);
    } else if (tid == 32) {
        for (int p = 0; p < n_pieces; ++p) {
            const int st = p % R;
            if (!mbar_wait(smem_addr(&bars[st]), (p / R) & 1, kLimitNs)) {
                atomicOr(status, 2u);
                break;
            }
            mbar_arrive(smem_addr(&bars[R + st]));
        }
    }
    __syncthreads();
}

__global__ void __launch_bounds__(256) fresh_kernel(float* states, unsigned* barrier, unsigned long long* out, int n,
                                                    unsigned* status) {
    float* mine = states + (size_t)blockIdx.x * 2048;
    for (int i = threadIdx.x; i < 2048; i += blockDim.x) mine[i] = (float)(blockIdx.x + i);
    __syncthreads();
    if (threadIdx.x == 0) {
        asm volatile("red.release.gpu.global.add.u32 [%0], %1;" :: "l"(barrier), "r"(1u) : "memory");
        const uint64_t t0 = global_ns();
        unsigned c;
        do {
            asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(c) : "l"(barrier) : "memory");
            if (global_ns() - t0 > kLimitNs) {
                atomicOr(status, 8u);
                break;
            }
        } while (c < (unsigned)n);
        out[3 * blockIdx.x + 2] = global_ns() - t0;
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        float v[20], acc = 0.f;
        const uint64_t t0 = global_ns();
#pragma unroll
        for (int t = 0; t < 20; ++t)
            v[t] = __ldcg(states + (size_t)((blockIdx.x + 7 * t + 1) % n) * 2048 + (blockIdx.x % 8) * 256 + lane);
#pragma unroll
        for (int t = 0; t < 20; ++t) acc += v[t];
        const uint64_t t1 = global_ns();
#pragma unroll
        for (int t = 0; t < 20; ++t)
            v[t] = __ldcg(states + (size_t)((blockIdx.x + 7 * t + 1) % n) * 2048 + (blockIdx.x % 8) * 256 + lane + 32);
#pragma unroll
        for (int t = 0; t < 20; ++t) acc += v[t];
        const uint64_t t2 = global_ns();
        if (lane == 0) {
            out[3 * blockIdx.x] = t1 - t0;
            out[3 * blockIdx.x + 1] = t2 - t1;
        }
        if (acc == -1.f) atomicOr(status, 16u);          // keeps the loads; never true for these values
    }
}

constexpr int kPushBytes = 96 * 1024;

__global__ void __launch_bounds__(256, 1) dsmem_kernel(unsigned long long* out) {
    extern __shared__ __align__(16) unsigned char buf[];
    const uint32_t rank = cluster_rank(), n = cluster_nrank();
    const uint32_t peer = (rank + 1) % n;
    cluster_sync();                                         // every CTA of the cluster is running
    const uint64_t t0 = global_ns();
    const uint32_t base = map_rank(smem_addr(buf), peer);
    for (int i = threadIdx.x; i < kPushBytes / 16; i += blockDim.x)
        st_cluster_v4(base + i * 16, make_uint4(i, rank, 0u, 0u));
    cluster_sync();                                         // every push has landed
    const uint64_t t1 = global_ns();
    if (threadIdx.x == 0) out[blockIdx.x] = t1 - t0;
}

static void run_dsmem(int cluster, unsigned long long* out) {
    const int ctas = 152 / cluster * cluster;
    cudaFuncSetAttribute(dsmem_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPushBytes);
    cudaFuncSetAttribute(dsmem_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(ctas);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = kPushBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    double sum = 0;
    const int reps = 4;
    for (int it = 0; it < reps; ++it) {
        if (cudaLaunchKernelEx(&cfg, dsmem_kernel, out) != cudaSuccess) {
            printf("dsmem cluster %d: launch failed (%s)\n", cluster, cudaGetErrorString(cudaGetLastError()));
            return;
        }
        cudaDeviceSynchronize();
        unsigned long long h[152];
        cudaMemcpy(h, out, ctas * 8, cudaMemcpyDeviceToHost);
        if (it == 0) continue;
        for (int i = 0; i < ctas; ++i) sum += h[i];
    }
    const double ns = sum / ((double)ctas * (reps - 1));
    printf("DSMEM push, clusters of %d (%3d CTAs): %.0f ns for %d KiB per CTA = %.1f GB/s per SM (%s)\n", cluster,
           ctas, ns, kPushBytes / 1024, kPushBytes / ns, cudaGetErrorString(cudaGetLastError()));
}

static PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 f = nullptr;
    if (!f) {
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", reinterpret_cast<void**>(&f), 12000,
                                             cudaEnableDefault, &q) != cudaSuccess)
            f = nullptr;
    }
    return f;
}

static bool map_kv(CUtensorMap* m, void* base, uint64_t rows) {
    cuuint64_t dims[2] = {kHd, rows};
    cuuint64_t strides[1] = {kHd * 2};
    cuuint32_t box[2] = {64, 128};
    cuuint32_t es[2] = {1, 1};
    auto enc = encoder();
    return enc && enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, base, dims, strides, box, es,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int R>
static void run_stream(const char* name, void* K, void* V, int n_kv, int ctas, int same_keys, unsigned* status) {
    CUtensorMap mk, mv;
    if (!map_kv(&mk, K, n_kv) || !map_kv(&mv, V, n_kv)) {
        printf("%s: tensor map encoding failed\n", name);
        return;
    }
    const int kpc = same_keys ? same_keys : (n_kv / ctas) / 128 * 128;
    const int smem = R * 32768 + 2048;
    cudaFuncSetAttribute(stream_kernel<R>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cudaEvent_t e0, e1;
    cudaEventCreate(&e0);
    cudaEventCreate(&e1);
    for (int i = 0; i < 2; ++i) stream_kernel<R><<<ctas, 64, smem>>>(mk, mv, kpc, same_keys != 0, status);
    const int iters = 5;
    cudaEventRecord(e0);
    for (int i = 0; i < iters; ++i) stream_kernel<R><<<ctas, 64, smem>>>(mk, mv, kpc, same_keys != 0, status);
    cudaEventRecord(e1);
    cudaEventSynchronize(e1);
    float ms = 0.f;
    cudaEventElapsedTime(&ms, e0, e1);
    unsigned st = 0;
    cudaMemcpy(&st, status, 4, cudaMemcpyDeviceToHost);
    const double bytes = 2.0 * (double)kpc * ctas * kHd * 2;
    printf("%-44s %3d CTAs, %d stages: %8.1f us per launch, %7.0f GB/s (status %u, %s)\n", name, ctas, R,
           ms * 1000.0 / iters, bytes / (ms / iters * 1e-3) / 1e9, st, cudaGetErrorString(cudaGetLastError()));
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
}

int main() {
    const int n_kv = 1 << 21;                               // 1 GiB each of K and V
    void *K = nullptr, *V = nullptr;
    unsigned* status = nullptr;
    if (cudaMalloc(&K, (size_t)n_kv * kHd * 2) != cudaSuccess || cudaMalloc(&V, (size_t)n_kv * kHd * 2) != cudaSuccess ||
        cudaMalloc(&status, 4) != cudaSuccess) {
        printf("allocation failed\n");
        return 1;
    }
    cudaMemset(K, 0, (size_t)n_kv * kHd * 2);
    cudaMemset(V, 0, (size_t)n_kv * kHd * 2);
    cudaMemset(status, 0, 4);
    run_stream<2>("stream K+V from HBM", K, V, n_kv, 152, 0, status);
    run_stream<4>("stream K+V from HBM", K, V, n_kv, 152, 0, status);
    run_stream<6>("stream K+V from HBM", K, V, n_kv, 152, 0, status);
    run_stream<6>("stream K+V from HBM", K, V, n_kv, 76, 0, status);
    run_stream<6>("same 8 MiB in every CTA (L2)", K, V, n_kv, 152, 8192, status);
    run_stream<6>("same 8 MiB in every CTA (L2)", K, V, n_kv, 76, 8192, status);

    const int n = 152;
    float* states = nullptr;
    unsigned* barrier = nullptr;
    unsigned long long* out = nullptr;
    cudaMalloc(&states, (size_t)n * 2048 * 4);
    cudaMalloc(&barrier, 4);
    cudaMalloc(&out, 3 * n * 8);
    double first = 0, again = 0, wait = 0;
    const int reps = 4;
    for (int it = 0; it < reps; ++it) {
        cudaMemset(barrier, 0, 4);
        fresh_kernel<<<n, 256>>>(states, barrier, out, n, status);
        cudaDeviceSynchronize();
        unsigned long long h[3 * 152];
        cudaMemcpy(h, out, sizeof(h), cudaMemcpyDeviceToHost);
        if (it == 0) continue;                              // first launch warms up
        for (int i = 0; i < n; ++i) {
            first += h[3 * i];
            again += h[3 * i + 1];
            wait += h[3 * i + 2];
        }
    }
    run_dsmem(2, out);
    run_dsmem(8, out);
    const double cnt = (double)n * (reps - 1);
    unsigned st = 0;
    cudaMemcpy(&st, status, 4, cudaMemcpyDeviceToHost);
    printf("after a grid barrier, 20 independent loads of lines other CTAs just wrote: %.0f ns; 20 more from the "
           "same blocks: %.0f ns; barrier wait %.0f ns (status %u, %s)\n",
           first / cnt, again / cnt, wait / cnt, st, cudaGetErrorString(cudaGetLastError()));
    return st == 0 ? 0 : 2;
}
