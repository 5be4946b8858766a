// Immersed-boundary samples ordered on the device ("GPU Optimization for High-Quality Kinetic
// Fluid Simulation", Sec. 4: samples sorted by l-block and by Morton code inside the block,
// Fig. 7), so that a moving body can replace its samples every step without a trip through
// the host.
//
// Each call places every sample (periodic axes wrap; a non-finite position or a stencil that
// would leave through a wall face drops the sample: weight 0, position 0, a key past every
// valid key, counted), sorts (key, index) pairs with a stable least-significant-digit radix
// sort over 8-bit digits, and gathers positions, boundary velocities and weights into the
// context's sample planes in that order.  Up to SMALL_N samples are ordered by one thread
// block in shared memory, key and index packed in one 64-bit word (one launch).  More take
// the multi-block sort: per digit pass a histogram per tile of SORT_TILE keys, one exclusive
// scan over (digit, tile), and a stable scatter.  Stability within a tile: each warp takes a
// contiguous share of the keys, 32 at a time, ranks them among the warp's lanes with the
// same digit (match_any), and the warps' digit counts are scanned in warp order.
#include <cstdint>
#include <utility>

#include "lbm_internal.h"

namespace lbm {
namespace {

using u64 = unsigned long long;

constexpr int SORT_THREADS = 256;
constexpr int SORT_WARPS = SORT_THREADS / 32;
constexpr int SORT_TILE = IB_SORT_TILE;           // keys per block, multi-block sort
constexpr int SORT_CHUNKS = SORT_TILE / SORT_WARPS / 32;   // 32-key chunks per warp
constexpr int SMALL_THREADS = 1024;
constexpr int SMALL_WARPS = SMALL_THREADS / 32;
constexpr int SMALL_N = 16384;                    // one block: 128 KiB of packed words
constexpr int SMALL_CHUNKS = SMALL_N / SMALL_THREADS;

struct OrderArgs {
    int n, dim, l;
    long long nbx, nby;
    u64 bad_key;                 // key of a dropped sample: past every valid key
    const float *xyz, *ub, *w;   // the caller's samples (device addresses)
};

__device__ unsigned digit_of(u64 k, int shift) { return (unsigned)(k >> shift) & 255u; }

// Key of sample s (bad_key for a dropped one).
__device__ u64 sample_key(const Params &P, const OrderArgs &A, int s, bool &valid)
{
    const float in[3] = {A.xyz[3 * s], A.dim > 1 ? A.xyz[3 * s + 1] : 0.0f,
                         A.dim > 2 ? A.xyz[3 * s + 2] : 0.0f};
    float x[3];
    valid = ib_place(P, A.dim, in, x);
    return valid ? ib_sort_key(x, A.dim, A.l, A.nbx, A.nby) : A.bad_key;
}

// Slot i of the context's sample planes (x3, ub3, w, kept) from the caller's sample src;
// returns whether the sample is kept.
__device__ bool put_sample(const Params &P, const OrderArgs &A, int i, int src)
{
    const float in[3] = {A.xyz[3 * src], A.dim > 1 ? A.xyz[3 * src + 1] : 0.0f,
                         A.dim > 2 ? A.xyz[3 * src + 2] : 0.0f};
    float x[3];
    const bool valid = ib_place(P, A.dim, in, x);
    float *planes = const_cast<float *>(P.ibx);
    const size_t cap = (size_t)P.ib_cap;
    for (int a = 0; a < 3; ++a) {
        planes[a * cap + i] = valid ? x[a] : 0.0f;
        planes[(3 + a) * cap + i] = (A.ub && a < A.dim) ? A.ub[3 * src + a] : 0.0f;
    }
    planes[6 * cap + i] = valid ? (A.w ? A.w[src] : 1.0f) : 0.0f;
    planes[7 * cap + i] = valid ? 1.0f : 0.0f;
    return valid;
}

// match_any over the lanes' digits (lanes without a key pass 256, which no key has) and
// each lane's rank among the lanes before it with the same digit.
__device__ void warp_rank(unsigned d, unsigned &peers, unsigned &rank)
{
    peers = __match_any_sync(0xffffffffu, d);
    rank = __popc(peers & ((1u << (threadIdx.x & 31u)) - 1u));
}

// ----------------------------------------------------------------- one block -------

// Words (key << vb) | index in shared memory; `passes` 8-bit digit passes over the key.
__global__ void __launch_bounds__(SMALL_THREADS) ib_order_small_kernel(const Params P,
                                                                        OrderArgs A, int vb,
                                                                        int passes, int *perm,
                                                                        unsigned *dropped)
{
    extern __shared__ u64 word[];
    __shared__ unsigned short cnt[SMALL_WARPS][256];
    __shared__ unsigned dbase[256];
    __shared__ unsigned n_drop;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) n_drop = 0;
    __syncthreads();
    for (int s = threadIdx.x; s < A.n; s += SMALL_THREADS) {
        bool valid;
        const u64 k = sample_key(P, A, s, valid);
        if (!valid) atomicAdd(&n_drop, 1u);
        word[s] = (k << vb) | (u64)s;
    }
    __syncthreads();
    // each warp owns a contiguous share of the words, 32 at a time
    const int per_warp = (A.n + SMALL_WARPS - 1) / SMALL_WARPS;
    const int lo = warp * per_warp, hi = min(A.n, lo + per_warp);
    for (int pass = 0; pass < passes; ++pass) {
        const int shift = vb + 8 * pass;
        u64 kk[SMALL_CHUNKS];
#pragma unroll
        for (int j = 0; j < SMALL_CHUNKS; ++j) {
            const int i = lo + 32 * j + lane;
            kk[j] = i < hi ? word[i] : 0ull;
        }
        for (int d = lane; d < 256; d += 32) cnt[warp][d] = 0;
        __syncwarp();
#pragma unroll
        for (int j = 0; j < SMALL_CHUNKS; ++j) {
            const int i = lo + 32 * j + lane;
            unsigned peers, rank;
            warp_rank(i < hi ? digit_of(kk[j], shift) : 256u, peers, rank);
            if (i < hi && rank == 0) cnt[warp][digit_of(kk[j], shift)] += __popc(peers);
            __syncwarp();
        }
        __syncthreads();
        if (threadIdx.x < 256) {        // warp-major offsets within each digit
            unsigned run = 0;
            for (int v = 0; v < SMALL_WARPS; ++v) {
                const unsigned c = cnt[v][threadIdx.x];
                cnt[v][threadIdx.x] = (unsigned short)run;
                run += c;
            }
            dbase[threadIdx.x] = run;
        }
        __syncthreads();
        if (warp == 0) {                // exclusive scan of the digit totals
            unsigned v[8], sum = 0;
            for (int k = 0; k < 8; ++k) {
                v[k] = dbase[8 * lane + k];
                sum += v[k];
            }
            unsigned incl = sum;
            for (int off = 1; off < 32; off <<= 1) {
                const unsigned t = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += t;
            }
            unsigned run = incl - sum;
            for (int k = 0; k < 8; ++k) {
                dbase[8 * lane + k] = run;
                run += v[k];
            }
        }
        __syncthreads();
#pragma unroll
        for (int j = 0; j < SMALL_CHUNKS; ++j) {
            const int i = lo + 32 * j + lane;
            const unsigned d = i < hi ? digit_of(kk[j], shift) : 256u;
            unsigned peers, rank;
            warp_rank(d, peers, rank);
            if (i < hi) word[dbase[d] + cnt[warp][d] + rank] = kk[j];
            __syncwarp();
            if (i < hi && rank == 0) cnt[warp][d] += __popc(peers);
            __syncwarp();
        }
        __syncthreads();
    }
    const u64 idx_mask = (1ull << vb) - 1ull;
    for (int i = threadIdx.x; i < A.n; i += SMALL_THREADS) {
        const int src = (int)(word[i] & idx_mask);
        perm[i] = src;
        put_sample(P, A, i, src);
    }
    if (threadIdx.x == 0) *dropped = n_drop;
}

// --------------------------------------------------------------- many blocks -------

__global__ void ib_key_kernel(const Params P, OrderArgs A, u64 *key, int *val, unsigned *dropped)
{
    const int s = blockIdx.x * blockDim.x + threadIdx.x;
    if (s >= A.n) return;
    bool valid;
    key[s] = sample_key(P, A, s, valid);
    val[s] = s;
    if (!valid) atomicAdd(dropped, 1u);
}

// Digit counts of one tile: hist[digit * tiles + tile].
__global__ void __launch_bounds__(SORT_THREADS) sort_hist_kernel(const u64 *key, int n, int shift,
                                                                 unsigned *hist, int tiles)
{
    __shared__ unsigned h[256];
    h[threadIdx.x] = 0;
    __syncthreads();
    for (int j = 0; j < SORT_TILE / SORT_THREADS; ++j) {
        const int i = blockIdx.x * SORT_TILE + j * SORT_THREADS + threadIdx.x;
        if (i < n) atomicAdd(&h[digit_of(key[i], shift)], 1u);
    }
    __syncthreads();
    hist[threadIdx.x * tiles + blockIdx.x] = h[threadIdx.x];
}

// Exclusive scan of a[0..len) in place, one block.
__global__ void __launch_bounds__(1024) sort_scan_kernel(unsigned *a, int len)
{
    __shared__ unsigned part[1024];
    const int chunk = (len + 1023) / 1024;
    const int lo = threadIdx.x * chunk, hi = min(len, lo + chunk);
    unsigned sum = 0;
    for (int i = lo; i < hi; ++i) sum += a[i];
    part[threadIdx.x] = sum;
    __syncthreads();
    for (int off = 1; off < 1024; off <<= 1) {
        const unsigned v = threadIdx.x >= off ? part[threadIdx.x - off] : 0u;
        __syncthreads();
        part[threadIdx.x] += v;
        __syncthreads();
    }
    unsigned run = part[threadIdx.x] - sum;
    for (int i = lo; i < hi; ++i) {
        const unsigned t = a[i];
        a[i] = run;
        run += t;
    }
}

// Stable scatter of one tile by the digit at `shift`.
__global__ void __launch_bounds__(SORT_THREADS) sort_scatter_kernel(const u64 *kin, const int *vin,
                                                                    u64 *kout, int *vout, int n,
                                                                    int shift,
                                                                    const unsigned *offs, int tiles)
{
    __shared__ unsigned cnt[SORT_WARPS][256];
    __shared__ unsigned base[256];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int lo = blockIdx.x * SORT_TILE + warp * (SORT_TILE / SORT_WARPS);
    const int hi = min(n, lo + SORT_TILE / SORT_WARPS);
    u64 kk[SORT_CHUNKS];
    int vv[SORT_CHUNKS];
#pragma unroll
    for (int j = 0; j < SORT_CHUNKS; ++j) {
        const int i = lo + 32 * j + lane;
        kk[j] = i < hi ? kin[i] : 0ull;
        vv[j] = i < hi ? vin[i] : 0;
    }
    for (int d = lane; d < 256; d += 32) cnt[warp][d] = 0;
    __syncwarp();
#pragma unroll
    for (int j = 0; j < SORT_CHUNKS; ++j) {
        const int i = lo + 32 * j + lane;
        unsigned peers, rank;
        warp_rank(i < hi ? digit_of(kk[j], shift) : 256u, peers, rank);
        if (i < hi && rank == 0) cnt[warp][digit_of(kk[j], shift)] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    {
        unsigned run = 0;
        for (int v = 0; v < SORT_WARPS; ++v) {
            const unsigned c = cnt[v][threadIdx.x];
            cnt[v][threadIdx.x] = run;
            run += c;
        }
        base[threadIdx.x] = offs[threadIdx.x * tiles + blockIdx.x];
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < SORT_CHUNKS; ++j) {
        const int i = lo + 32 * j + lane;
        const unsigned d = i < hi ? digit_of(kk[j], shift) : 256u;
        unsigned peers, rank;
        warp_rank(d, peers, rank);
        if (i < hi) {
            const unsigned pos = base[d] + cnt[warp][d] + rank;
            kout[pos] = kk[j];
            vout[pos] = vv[j];
        }
        __syncwarp();
        if (i < hi && rank == 0) cnt[warp][d] += __popc(peers);
        __syncwarp();
    }
}

// Slot i from caller sample val[i]; perm_out (optional) records the order, dropped (optional)
// counts the samples not kept.
__global__ void ib_gather_kernel(const Params P, OrderArgs A, const int *val, int *perm_out,
                                 unsigned *dropped)
{
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= A.n) return;
    const int src = val[i];
    if (perm_out) perm_out[i] = src;
    if (!put_sample(P, A, i, src) && dropped) atomicAdd(dropped, 1u);
}

int bit_length(u64 v)
{
    int b = 0;
    while (v) {
        ++b;
        v >>= 1;
    }
    return b;
}

}  // namespace

cudaError_t launch_ib_order(int lattice, const Params &P, int n, int l, const float *xyz,
                            const float *ub, const float *w, void *scratch, bool reorder,
                            cudaStream_t s)
{
    if (n <= 0) return cudaSuccess;
    OrderArgs A;
    A.n = n;
    A.dim = lattice == 9 ? 2 : 3;
    A.l = l;
    A.nbx = (P.nx + l - 1) / l;
    A.nby = (P.ny + l - 1) / l;
    const long long nbz = A.dim == 3 ? (P.nz + l - 1) / l : 1;
    const u64 blocks = (u64)A.nbx * (u64)A.nby * (u64)nbz;
    A.bad_key = blocks << IB_MORTON_BITS;
    A.xyz = xyz;
    A.ub = ub;
    A.w = w;
    const int key_bits = IB_MORTON_BITS + bit_length(blocks);
    const int passes = (key_bits + 7) / 8;
    // scratch: keys[2][cap], vals[2][cap], hist[256 * tiles], the dropped-sample count
    const size_t cap = (size_t)P.ib_cap;
    const int tiles = (n + SORT_TILE - 1) / SORT_TILE;
    u64 *key0 = static_cast<u64 *>(scratch), *key1 = key0 + cap;
    int *val0 = reinterpret_cast<int *>(key1 + cap), *val1 = val0 + cap;
    unsigned *hist = reinterpret_cast<unsigned *>(val1 + cap);
    int *perm = ib_order_perm(P, scratch);
    unsigned *dropped = ib_dropped_counter(P, scratch);
    cudaError_t e = cudaSuccess;
    if (!reorder) {   // the order of the last sort
        if ((e = cudaMemsetAsync(dropped, 0, sizeof(unsigned), s)) != cudaSuccess) return e;
        ib_gather_kernel<<<(n + 255) / 256, 256, 0, s>>>(P, A, perm, nullptr, dropped);
        return cudaGetLastError();
    }
    const int vb = bit_length((u64)(n - 1)) > 0 ? bit_length((u64)(n - 1)) : 1;
    if (n <= SMALL_N && key_bits + vb <= 64) {
        const int smem = SMALL_N * (int)sizeof(u64);
        e = cudaFuncSetAttribute(ib_order_small_kernel,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        ib_order_small_kernel<<<1, SMALL_THREADS, smem, s>>>(P, A, vb, passes, perm, dropped);
        return cudaGetLastError();
    }
    if ((e = cudaMemsetAsync(dropped, 0, sizeof(unsigned), s)) != cudaSuccess) return e;
    ib_key_kernel<<<(n + 255) / 256, 256, 0, s>>>(P, A, key0, val0, dropped);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    for (int pass = 0; pass < passes; ++pass) {
        const int shift = 8 * pass;
        sort_hist_kernel<<<tiles, SORT_THREADS, 0, s>>>(key0, n, shift, hist, tiles);
        sort_scan_kernel<<<1, 1024, 0, s>>>(hist, 256 * tiles);
        sort_scatter_kernel<<<tiles, SORT_THREADS, 0, s>>>(key0, val0, key1, val1, n, shift,
                                                          hist, tiles);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        std::swap(key0, key1);
        std::swap(val0, val1);
    }
    ib_gather_kernel<<<(n + 255) / 256, 256, 0, s>>>(P, A, val0, perm, nullptr);
    return cudaGetLastError();
}

}  // namespace lbm
