// lbm_reduce_populations_static: a population reduction that allocates nothing.
//
// Some callers cannot call cudaMalloc at all: code that runs inside another framework's
// memory pool, in a process where the allocator is owned by someone else, or in a
// real-time loop where an allocation (and the synchronisation it can imply) is not
// allowed.  They cannot give the library a workspace either.  For them this entry point
// sums mass, momentum and thermal energy of populations held in memory the caller owns,
// with its reduction scratch in a file-scope static device array instead of a workspace.
//
// The scratch holds one row of partial sums per thread block; every block writes its
// row before the finishing kernel reads it (stream order), so nothing in it needs to be
// cleared between calls.  All calls share the one array: calls that overlap on the GPU
// (on different streams, or from different threads without ordering) race on it.
#include <cstdint>
#include <mutex>
#include <string>

#include "../../include/lbm.h"
#include "lbm_internal.h"

namespace {

constexpr int RED_THREADS = 256;
constexpr long long RED_CELLS_PER_BLOCK = 8192;      // 32 cells per thread
constexpr int RED_MAX_BLOCKS = 32768;                // 2 MiB of scratch
constexpr int RED_ROW = 8;                           // doubles per partial row
constexpr long long RED_MAX_CELLS = RED_CELLS_PER_BLOCK * RED_MAX_BLOCKS;  // 2^28
constexpr int MAX_DEVICES = 64;

static __device__ __align__(256) double g_reduce_scratch[RED_MAX_BLOCKS * RED_ROW];

std::mutex g_setup_mutex;
double *g_scratch_address[MAX_DEVICES] = {};

// Sums of one tile of cells: [0] sum f, [1..3] sum c f, [4] sum g, [5] non-finite cells.
template <class L, class TL>
__global__ void __launch_bounds__(RED_THREADS) reduce_tile_kernel(const float *__restrict__ f,
                                                                  const float *__restrict__ g,
                                                                  long long N, double *scratch)
{
    double acc[6] = {0, 0, 0, 0, 0, 0};
    const long long begin = blockIdx.x * RED_CELLS_PER_BLOCK;
    const long long end = begin + RED_CELLS_PER_BLOCK < N ? begin + RED_CELLS_PER_BLOCK : N;
    for (long long i = begin + threadIdx.x; i < end; i += RED_THREADS) {
        float m = 0.0f, jx = 0.0f, jy = 0.0f, jz = 0.0f, t = 0.0f;
#pragma unroll
        for (int q = 0; q < L::Q; ++q) {
            const float v = f[q * N + i];
            m += v;
            if (L::cx(q)) jx += L::cx(q) * v;
            if (L::cy(q)) jy += L::cy(q) * v;
            if (L::cz(q)) jz += L::cz(q) * v;
        }
        if constexpr (TL::Q > 0) {
#pragma unroll
            for (int k = 0; k < TL::Q; ++k) t += g[k * N + i];
        }
        acc[0] += m;
        acc[1] += jx;
        acc[2] += jy;
        acc[3] += jz;
        acc[4] += t;
        if (!isfinite(m) || !isfinite(t)) acc[5] += 1.0;
    }
    __shared__ double sh[RED_THREADS / 32][6];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int k = 0; k < 6; ++k) {
        double v = acc[k];
        for (int s = 16; s > 0; s >>= 1) v += __shfl_down_sync(0xffffffffu, v, s);
        if (lane == 0) sh[warp][k] = v;
    }
    __syncthreads();
    if (threadIdx.x < 6) {
        double v = 0.0;
        for (int w = 0; w < RED_THREADS / 32; ++w) v += sh[w][threadIdx.x];
        scratch[blockIdx.x * RED_ROW + threadIdx.x] = v;
    }
}

// Sum the rows of the scratch in a fixed order into out[0..5].
__global__ void __launch_bounds__(RED_THREADS) reduce_rows_kernel(const double *scratch,
                                                                  int rows, double *out)
{
    __shared__ double sh[RED_THREADS][6];
    double acc[6] = {0, 0, 0, 0, 0, 0};
    for (int r = threadIdx.x; r < rows; r += RED_THREADS)
        for (int k = 0; k < 6; ++k) acc[k] += scratch[r * RED_ROW + k];
    for (int k = 0; k < 6; ++k) sh[threadIdx.x][k] = acc[k];
    __syncthreads();
    for (int s = RED_THREADS / 2; s > 0; s >>= 1) {
        if (threadIdx.x < s)
            for (int k = 0; k < 6; ++k) sh[threadIdx.x][k] += sh[threadIdx.x + s][k];
        __syncthreads();
    }
    if (threadIdx.x < 6) out[threadIdx.x] = sh[0][threadIdx.x];
}

lbm_status reject(lbm_status s, const std::string &msg)
{
    lbm_internal_set_error(msg.c_str());
    return s;
}

// Device address of a caller pointer: device memory of `dev`, or page-locked host.
bool usable(const void *p, int dev, void **out)
{
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if ((a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) && a.device == dev) {
        *out = const_cast<void *>(p);
        return true;
    }
    if (a.type == cudaMemoryTypeHost) {
        *out = a.devicePointer ? a.devicePointer : const_cast<void *>(p);
        return true;
    }
    return false;
}

template <class L, class TL>
cudaError_t launch(const float *f, const float *g, long long N, double *scratch, double *out,
                   cudaStream_t s)
{
    const int blocks = (int)((N + RED_CELLS_PER_BLOCK - 1) / RED_CELLS_PER_BLOCK);
    reduce_tile_kernel<L, TL><<<blocks, RED_THREADS, 0, s>>>(f, g, N, scratch);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    reduce_rows_kernel<<<1, RED_THREADS, 0, s>>>(scratch, blocks, out);
    return cudaGetLastError();
}

}  // namespace

extern "C" lbm_status lbm_reduce_populations_static(int lattice, int thermal, int nx, int ny,
                                                    int nz, const float *f, const float *g,
                                                    double *out, void *cuda_stream)
{
    if (lattice != LBM_D3Q19 && lattice != LBM_D2Q9 && lattice != LBM_D3Q27)
        return reject(LBM_ERR_ARG, "lattice must be LBM_D3Q19, LBM_D2Q9 or LBM_D3Q27");
    if (thermal != LBM_THERMAL_NONE && !((lattice == LBM_D3Q19 && thermal == LBM_D3Q7) ||
                                         (lattice == LBM_D2Q9 && thermal == LBM_D2Q5)))
        return reject(LBM_ERR_ARG, "thermal lattice must be none, D3Q7 (D3Q19) or D2Q5 (D2Q9)");
    if (nx < 1 || ny < 1 || nz < 1) return reject(LBM_ERR_ARG, "grid sizes must be >= 1");
    if (lattice == LBM_D2Q9 && nz != 1) return reject(LBM_ERR_ARG, "D2Q9 needs nz == 1");
    // nx*ny < 2^62 cannot overflow; once it is within the limit, so is the product with nz
    const long long nxy = (long long)nx * ny;
    if (nxy > RED_MAX_CELLS || nxy * nz > RED_MAX_CELLS)
        return reject(LBM_ERR_ARG, "lbm_reduce_populations_static: " + std::to_string(nx) +
                                       "x" + std::to_string(ny) + "x" + std::to_string(nz) +
                                       " cells exceed the static scratch limit of " +
                                       std::to_string(RED_MAX_CELLS) + " cells");
    const long long N = nxy * nz;
    if (!f || !out || (thermal && !g))
        return reject(LBM_ERR_ARG, "f, out (and g with a thermal lattice) are required");
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= MAX_DEVICES)
        return reject(LBM_ERR_CUDA, "no usable current device");
    double *scratch = nullptr;
    {
        // once per device, with that device current: the scratch array's device address
        std::lock_guard<std::mutex> lock(g_setup_mutex);
        if (!g_scratch_address[dev]) {
            e = cudaGetSymbolAddress(reinterpret_cast<void **>(&scratch), g_reduce_scratch);
            if (e != cudaSuccess)
                return reject(LBM_ERR_CUDA, std::string("cudaGetSymbolAddress: ") +
                                                cudaGetErrorString(e));
            g_scratch_address[dev] = scratch;
        }
        scratch = g_scratch_address[dev];
    }
    void *df = nullptr, *dg = nullptr, *dout = nullptr;
    if (!usable(f, dev, &df) || (thermal && !usable(g, dev, &dg)) || !usable(out, dev, &dout))
        return reject(LBM_ERR_ARG,
                      "f, g and out must be device memory of the current device or page-locked "
                      "host memory");
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    const float *pf = static_cast<const float *>(df), *pg = static_cast<const float *>(dg);
    double *po = static_cast<double *>(dout);
    if (lattice == LBM_D3Q27)
        e = launch<lbm::D3Q27, lbm::NoThermal>(pf, pg, N, scratch, po, s);
    else if (lattice == LBM_D3Q19)
        e = thermal ? launch<lbm::D3Q19, lbm::D3Q7>(pf, pg, N, scratch, po, s)
                    : launch<lbm::D3Q19, lbm::NoThermal>(pf, pg, N, scratch, po, s);
    else
        e = thermal ? launch<lbm::D2Q9, lbm::D2Q5>(pf, pg, N, scratch, po, s)
                    : launch<lbm::D2Q9, lbm::NoThermal>(pf, pg, N, scratch, po, s);
    if (e != cudaSuccess)
        return reject(LBM_ERR_CUDA, std::string("reduction kernels: ") + cudaGetErrorString(e));
    return LBM_OK;
}
