// C ABI of the GB300 lattice-Boltzmann library (declared in include/lbm.h): argument
// validation, workspace layout, parity bookkeeping, launches and error status.
#include <cmath>
#include <cstdio>
#include <cstring>
#include <new>
#include <array>
#include <string>
#include <utility>
#include <algorithm>
#include <vector>

#include "../../include/lbm.h"
#include "lbm_internal.h"
#include "lbm_halo.h"
#include "lbm_setup.h"

using lbm_setup::Layout;
using lbm_setup::ALIGN;

namespace {

thread_local std::string g_error;  // errors without a context (create, workspace_bytes)

struct DeviceGuard {
    int prev = -1;
    bool changed = false;
    explicit DeviceGuard(int dev)
    {
        if (cudaGetDevice(&prev) == cudaSuccess && prev != dev) {
            changed = cudaSetDevice(dev) == cudaSuccess;
        }
    }
    ~DeviceGuard()
    {
        if (changed) cudaSetDevice(prev);
    }
};

}  // namespace

struct lbm_ctx {
    lbm_config cfg{};
    Layout L;
    lbm::Params P{};
    char *ws = nullptr;
    uint8_t *solid = nullptr;
    double *partial = nullptr, *result = nullptr;
    cudaStream_t stream = nullptr;
    int device = 0;
    bool chained = false;   // step kernels launched chained (lbm::chain_steps)
    int parity = 0;
    long long steps = 0;
    bool initialized = false;
    // lbm_step_planes: outer-axis planes already stepped in the current (unfinished) step
    // boxes of cells stepped so far in a step split across lbm_step_box calls, and the
    // cells still to step (> 0 while a step is partly done)
    std::vector<std::array<int, 6>> boxes_done;
    long long cells_left = 0;
    int ib_order_n = -1;   // sample count of the stored sample order, -1 = none
    std::string err;
    // CUDA graphs of GRAPH_STEPS steps, one per start parity, built on first use for
    // grids small enough that launch overhead matters; captured on a private stream.
    cudaGraphExec_t graph[2] = {nullptr, nullptr};
    cudaStream_t capture_stream = nullptr;
    bool graphs_disabled = false;
    void drop_graphs()
    {
        for (auto &g : graph)
            if (g) cudaGraphExecDestroy(g);
        graph[0] = graph[1] = nullptr;
    }
    ~lbm_ctx()
    {
        drop_graphs();
        if (capture_stream) cudaStreamDestroy(capture_stream);
    }
};

namespace {

lbm_status fail(lbm_ctx *c, lbm_status s, const std::string &msg)
{
    if (c) c->err = msg;
    else g_error = msg;
    return s;
}

// Calls that need a whole time step behind them, made while lbm_step_planes has stepped
// only some of the planes.
lbm_status partly_stepped(lbm_ctx *c)
{
    return fail(c, LBM_ERR_STATE,
                "a step is partly done: lbm_step_box (or lbm_step_planes) must cover the "
                "remaining cells first");
}

lbm_status cuda_fail(lbm_ctx *c, cudaError_t e, const char *where)
{
    std::string m = std::string(where) + ": " + cudaGetErrorName(e) + " (" +
                    cudaGetErrorString(e) + ")";
    return fail(c, LBM_ERR_CUDA, m);
}

// Resolve a caller's field pointer to an address a kernel can use.
lbm_status device_address(lbm_ctx *c, const void *p, const char *what, void **out)
{
    cudaPointerAttributes a;
    cudaError_t e = cudaPointerGetAttributes(&a, p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(c, LBM_ERR_ARG, std::string(what) + ": not a valid pointer");
    }
    switch (a.type) {
    case cudaMemoryTypeDevice:
    case cudaMemoryTypeManaged:
        if (a.device != c->device)
            return fail(c, LBM_ERR_ARG, std::string(what) + ": memory of another device");
        *out = const_cast<void *>(p);
        return LBM_OK;
    case cudaMemoryTypeHost:
        *out = a.devicePointer ? a.devicePointer : const_cast<void *>(p);
        return LBM_OK;
    default: {
        int pageable = 0;
        cudaDeviceGetAttribute(&pageable, cudaDevAttrPageableMemoryAccess, c->device);
        if (!pageable)
            return fail(c, LBM_ERR_ARG,
                        std::string(what) +
                            ": pageable host memory; pass device or page-locked memory");
        *out = const_cast<void *>(p);
        return LBM_OK;
    }
    }
}

// Read pattern of the stored logical state.
int pattern(const lbm_ctx *c)
{
    if (c->L.streaming == LBM_STREAM_PULL) return lbm::PULL;
    if (c->L.streaming == LBM_STREAM_SPLIT) return lbm::NATURAL;
    return c->parity ? lbm::AA_ODD : lbm::NATURAL;
}

}  // namespace

void lbm_internal_set_error(const char *msg) { g_error = msg ? msg : ""; }

extern "C" {

lbm_status lbm_workspace_bytes(const lbm_config *cfg, size_t *bytes)
{
    if (!bytes) return fail(nullptr, LBM_ERR_ARG, "bytes is NULL");
    Layout L;
    std::string why;
    lbm_status s = lbm_setup::validate(cfg, &L, &why);
    if (s != LBM_OK) return fail(nullptr, s, why);
    *bytes = L.bytes;
    return LBM_OK;
}

lbm_status lbm_create(const lbm_config *cfg, void *d_workspace, size_t workspace_bytes,
                      void *cuda_stream, lbm_ctx **out)
{
    if (!out) return fail(nullptr, LBM_ERR_ARG, "out is NULL");
    *out = nullptr;
    Layout L;
    std::string why;
    lbm_status s = lbm_setup::validate(cfg, &L, &why);
    if (s != LBM_OK) return fail(nullptr, s, why);
    if (!d_workspace) return fail(nullptr, LBM_ERR_WORKSPACE, "workspace is NULL");
    if (reinterpret_cast<uintptr_t>(d_workspace) % ALIGN)
        return fail(nullptr, LBM_ERR_WORKSPACE, "workspace must be 256-byte aligned");
    if (workspace_bytes < L.bytes)
        return fail(nullptr, LBM_ERR_WORKSPACE,
                    "workspace too small: need " + std::to_string(L.bytes) + " bytes");
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(nullptr, e, "cudaGetDevice");
    cudaPointerAttributes a;
    e = cudaPointerGetAttributes(&a, d_workspace);
    if (e != cudaSuccess || a.type != cudaMemoryTypeDevice || a.device != dev) {
        cudaGetLastError();
        return fail(nullptr, LBM_ERR_WORKSPACE,
                    "workspace must be device memory of the current device");
    }
    lbm_ctx *c = new (std::nothrow) lbm_ctx();
    if (!c) return fail(nullptr, LBM_ERR_ARG, "out of host memory");
    c->cfg = *cfg;
    c->cfg.solid_mask = nullptr;
    c->L = L;
    c->ws = static_cast<char *>(d_workspace);
    c->stream = static_cast<cudaStream_t>(cuda_stream);
    c->device = dev;
    {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            cudaGetLastError();
        const lbm::Shape sh = lbm::cell_shape(cfg->nx, cfg->ny, cfg->nz);
        c->chained = sms > 0 && lbm::chain_steps((long long)sh.grid.x * sh.grid.y * sh.grid.z, sms);
    }
    c->partial = reinterpret_cast<double *>(c->ws + L.off_partial);
    c->result = reinterpret_cast<double *>(c->ws + L.off_result);
    lbm_setup::fill_params(c->cfg, c->L, c->ws, c->P);
    if (L.ib_cap > 0) {
        e = cudaMemsetAsync(c->P.fib, 0, 3 * L.S * sizeof(float), c->stream);

        if (e != cudaSuccess) {
            lbm_status r = cuda_fail(nullptr, e, "clearing the immersed-boundary force");
            delete c;
            return r;
        }
    }
    if (L.masked) {
        uint8_t *solid = nullptr;
        if (L.has_solid) {
            solid = reinterpret_cast<uint8_t *>(c->ws + L.off_solid);
            e = cudaMemcpyAsync(solid, cfg->solid_mask, (size_t)L.N, cudaMemcpyHostToDevice,
                                c->stream);
            if (e != cudaSuccess) {
                lbm_status r = cuda_fail(nullptr, e, "copy of solid_mask");
                delete c;
                return r;
            }
        }
        e = lbm::launch_mask(cfg->lattice, cfg->thermal, c->P, solid,
                             const_cast<uint32_t *>(c->P.mask), c->stream);
        if (e != cudaSuccess) {
            lbm_status r = cuda_fail(nullptr, e, "mask kernel");
            delete c;
            return r;
        }
    }
    *out = c;
    return LBM_OK;
}

lbm_status lbm_init_equilibrium(lbm_ctx *c, const float *rho, const float *u, const float *T)
{
    if (!c) return fail(nullptr, LBM_ERR_ARG, "ctx is NULL");
    if (c->cells_left) return partly_stepped(c);
    if (!rho || !u) return fail(c, LBM_ERR_ARG, "rho and u are required");
    if (c->L.QT && !T) return fail(c, LBM_ERR_ARG, "T is required with a thermal lattice");
    DeviceGuard guard(c->device);
    void *dr, *du, *dT = nullptr;
    lbm_status s = device_address(c, rho, "rho", &dr);
    if (s == LBM_OK) s = device_address(c, u, "u", &du);
    if (s == LBM_OK && c->L.QT) s = device_address(c, T, "T", &dT);
    if (s != LBM_OK) return s;
    // the AA state starts at parity 0 (natural slots); SPLIT stores the natural state;
    // PULL stores a post-collision state read with the pull pattern.  Parity 0 always
    // means the first population buffer is current (the step graphs rely on it).
    c->parity = 0;
    const int ib_n = c->P.ib_n;
    lbm_setup::fill_params(c->cfg, c->L, c->ws, c->P);
    c->P.ib_n = ib_n;
    const int pat = (c->L.streaming == LBM_STREAM_PULL) ? lbm::PULL : lbm::NATURAL;
    cudaError_t e = lbm::launch_init(c->cfg.lattice, c->cfg.thermal, pat, c->P,
                                     (const float *)dr, (const float *)du, (const float *)dT,
                                     c->stream);
    if (e != cudaSuccess) return cuda_fail(c, e, "init kernel");
    c->parity = 0;
    c->steps = 0;
    c->initialized = true;
    return LBM_OK;
}

namespace {

constexpr int GRAPH_STEPS = 64;                    // even: parity and buffers come back
constexpr long long GRAPH_MAX_CELLS = 1LL << 22;   // launch-bound below ~4 M cells

// Enqueue one step on `stream` from the state (P, parity) and advance them.
cudaError_t enqueue_step(const lbm_ctx *c, lbm::Params &P, int &parity, cudaStream_t stream)
{
    const lbm::Shape sh = lbm::cell_shape(c->cfg.nx, c->cfg.ny, c->cfg.nz);
    const int whole_lo[3] = {0, 0, 0}, whole_hi[3] = {c->cfg.nx, c->cfg.ny, c->cfg.nz};
    const lbm::Shape sh_aa =
        lbm::step_shape(c->cfg.nx, c->cfg.ny, c->cfg.nz, c->L.dim, whole_lo, whole_hi, P.linear);
    // 32-bit population indices when the largest index (Q * S - 1) fits
    const bool narrow = (unsigned long long)c->L.Q * c->L.S <= 0xffffffffull;
    const bool d3 = c->cfg.lattice == LBM_D3Q19;
    const int th = c->cfg.thermal, coll = c->cfg.collision;
    const int masked = !c->L.masked ? 0 : (c->L.ib_cap > 0 ? 2 : 1);
    cudaError_t e;
    if (P.ib_n > 0) {
        const int pat = c->L.streaming == LBM_STREAM_PULL    ? lbm::PULL
                        : c->L.streaming == LBM_STREAM_SPLIT ? lbm::NATURAL
                        : parity                             ? lbm::AA_ODD
                                                             : lbm::NATURAL;
        e = lbm::launch_ib(c->cfg.lattice, th, pat, P, stream, c->chained);
        if (e != cudaSuccess) return e;
    }
    switch (c->L.streaming) {
    case LBM_STREAM_PULL:
        e = d3 ? lbm::launch_pull_d3q19(th, coll, masked, narrow, P, sh, stream, c->chained)
               : lbm::launch_pull_d2q9(th, coll, masked, narrow, P, sh, stream, c->chained);
        break;
    case LBM_STREAM_SPLIT:
        e = d3 ? lbm::launch_split_d3q19(th, coll, masked, narrow, P, sh, stream, c->chained)
               : lbm::launch_split_d2q9(th, coll, masked, narrow, P, sh, stream, c->chained);
        break;
    default:
        if (c->cfg.lattice == LBM_D3Q27)
            e = lbm::launch_step_d3q27(masked, parity != 0, narrow, P, sh_aa, stream, c->chained);
        else
            e = d3 ? lbm::launch_step_d3q19(th, coll, masked, parity != 0, narrow, P, sh_aa,
                                            stream, c->chained)
                   : lbm::launch_step_d2q9(th, coll, masked, parity != 0, narrow, P, sh_aa,
                                           stream, c->chained);
    }
    if (c->L.streaming != LBM_STREAM_AA) {
        std::swap(P.f, P.fo);
        std::swap(P.g, P.go);
    }
    parity ^= 1;
    return e;
}

// AA step kernel launch over the box of cells [lo, hi) (lbm_step_box).
cudaError_t launch_box(const lbm_ctx *c, const lbm::Params &P0, int parity, const int lo[3],
                       const int hi[3], cudaStream_t stream, bool chained)
{
    const bool d2 = c->cfg.lattice == LBM_D2Q9;
    lbm::Params P = P0;
    bool linear = false;
    const lbm::Shape sh =
        lbm::step_shape(c->cfg.nx, c->cfg.ny, c->cfg.nz, c->L.dim, lo, hi, P0.linear, &linear);
    P.linear = linear;
    for (int a = 0; a < 3; ++a) {
        P.run_lo[a] = lo[a];
        P.run_hi[a] = hi[a];
    }
    const bool narrow = (unsigned long long)c->L.Q * c->L.S <= 0xffffffffull;
    const int th = c->cfg.thermal, coll = c->cfg.collision;
    const int masked = !c->L.masked ? 0 : (c->L.ib_cap > 0 ? 2 : 1);
    const bool odd = parity != 0;
    if (c->cfg.lattice == LBM_D3Q27)
        return lbm::launch_step_d3q27(masked, odd, narrow, P, sh, stream, chained, true);
    return d2 ? lbm::launch_step_d2q9(th, coll, masked, odd, narrow, P, sh, stream, chained, true)
              : lbm::launch_step_d3q19(th, coll, masked, odd, narrow, P, sh, stream, chained,
                                       true);
}

// The graph of GRAPH_STEPS steps starting at the context's parity (built on first use).
// Returns nullptr (and stops trying) if capture is not possible.
cudaGraphExec_t step_graph(lbm_ctx *c)
{
    if (c->graphs_disabled) return nullptr;
    cudaGraphExec_t &exec = c->graph[c->parity];
    if (exec) return exec;
    if (!c->capture_stream &&
        cudaStreamCreateWithFlags(&c->capture_stream, cudaStreamNonBlocking) != cudaSuccess) {
        cudaGetLastError();
        c->graphs_disabled = true;
        return nullptr;
    }
    cudaGraph_t graph = nullptr;
    bool ok = cudaStreamBeginCapture(c->capture_stream, cudaStreamCaptureModeRelaxed) ==
              cudaSuccess;
    lbm::Params P = c->P;
    int parity = c->parity;
    for (int i = 0; ok && i < GRAPH_STEPS; ++i)
        ok = enqueue_step(c, P, parity, c->capture_stream) == cudaSuccess;
    const cudaError_t end = cudaStreamEndCapture(c->capture_stream, &graph);
    ok = ok && end == cudaSuccess && graph &&
         cudaGraphInstantiate(&exec, graph, 0) == cudaSuccess;
    if (graph) cudaGraphDestroy(graph);
    if (!ok) {
        cudaGetLastError();
        exec = nullptr;
        c->graphs_disabled = true;
    }
    return exec;
}

}  // namespace

lbm_status lbm_step(lbm_ctx *c, int n)
{
    if (!c) return fail(nullptr, LBM_ERR_ARG, "ctx is NULL");
    if (n < 0) return fail(c, LBM_ERR_ARG, "n must be >= 0");
    if (!c->initialized) return fail(c, LBM_ERR_STATE, "no state: call lbm_init_equilibrium");
    if (c->cells_left) return partly_stepped(c);
    DeviceGuard guard(c->device);
    // Small grids: replay a captured graph of GRAPH_STEPS steps (it leaves the parity and
    // the buffers as it found them), then launch the remainder one by one.
    if (c->L.N <= GRAPH_MAX_CELLS && n >= GRAPH_STEPS) {
        while (n >= GRAPH_STEPS) {
            cudaGraphExec_t exec = step_graph(c);
            if (!exec) break;
            cudaError_t e = cudaGraphLaunch(exec, c->stream);
            if (e != cudaSuccess) return cuda_fail(c, e, "step graph");
            c->steps += GRAPH_STEPS;
            n -= GRAPH_STEPS;
        }
    }
    for (int i = 0; i < n; ++i) {
        cudaError_t e = enqueue_step(c, c->P, c->parity, c->stream);
        if (e != cudaSuccess) return cuda_fail(c, e, "step kernel");
        ++c->steps;
    }
    return LBM_OK;
}

lbm_status lbm_step_box(lbm_ctx *c, const int *lo, const int *hi)
{
    if (!c) return fail(nullptr, LBM_ERR_ARG, "ctx is NULL");
    if (!lo || !hi) return fail(c, LBM_ERR_ARG, "lo and hi are required");
    if (!c->initialized) return fail(c, LBM_ERR_STATE, "no state: call lbm_init_equilibrium");
    if (c->L.streaming != LBM_STREAM_AA)
        return fail(c, LBM_ERR_UNSUPPORTED, "stepping part of the grid needs the AA layout");
    if (c->L.ib_cap > 0)
        return fail(c, LBM_ERR_UNSUPPORTED,
                    "stepping part of the grid takes no context with immersed-boundary capacity");
    const int n[3] = {c->cfg.nx, c->cfg.ny, c->cfg.nz};
    for (int a = 0; a < 3; ++a)
        if (lo[a] < 0 || hi[a] > n[a] || lo[a] >= hi[a])
            return fail(c, LBM_ERR_ARG, "the box [lo, hi) must be non-empty and inside the grid "
                                        "on every axis");
    // boxes of one step may not overlap: each cell is stepped once
    for (const auto &b : c->boxes_done) {
        bool meet = true;
        for (int a = 0; a < 3; ++a) meet = meet && lo[a] < b[3 + a] && b[a] < hi[a];
        if (meet) return fail(c, LBM_ERR_ARG, "the box overlaps one already stepped in this step");
    }
    if (!c->cells_left) {
        c->boxes_done.clear();
        c->cells_left = (long long)n[0] * n[1] * n[2];
    }
    DeviceGuard guard(c->device);
    // not chained: the launch may follow an event wait on another stream's halo work
    cudaError_t e = launch_box(c, c->P, c->parity, lo, hi, c->stream, false);
    if (e != cudaSuccess) return cuda_fail(c, e, "step kernel (box)");
    c->boxes_done.push_back({lo[0], lo[1], lo[2], hi[0], hi[1], hi[2]});
    c->cells_left -= (long long)(hi[0] - lo[0]) * (hi[1] - lo[1]) * (hi[2] - lo[2]);
    if (!c->cells_left) {
        c->boxes_done.clear();
        c->parity ^= 1;
        ++c->steps;
    }
    return LBM_OK;
}

lbm_status lbm_step_planes(lbm_ctx *c, int lo, int hi)
{
    if (!c) return fail(nullptr, LBM_ERR_ARG, "ctx is NULL");
    const int outer = c->L.dim - 1;
    int blo[3] = {0, 0, 0}, bhi[3] = {c->cfg.nx, c->cfg.ny, c->cfg.nz};
    blo[outer] = lo;
    bhi[outer] = hi;
    return lbm_step_box(c, blo, bhi);
}

lbm_status lbm_macroscopic(lbm_ctx *c, float *rho, float *u, float *T)
{
    if (!c) return fail(nullptr, LBM_ERR_ARG, "ctx is NULL");
    if (!c->initialized) return fail(c, LBM_ERR_STATE, "no state: call lbm_init_equilibrium");
    if (c->cells_left) return partly_stepped(c);
    DeviceGuard guard(c->device);
    void *dr = nullptr, *du = nullptr, *dT = nullptr;
    lbm_status s = LBM_OK;
    if (rho) s = device_address(c, rho, "rho", &dr);
    if (s == LBM_OK && u) s = device_address(c, u, "u", &du);
    if (s == LBM_OK && T && c->L.QT) s = device_address(c, T, "T", &dT);
    if (s != LBM_OK) return s;
    cudaError_t e = lbm::launch_macro(c->cfg.lattice, c->cfg.thermal, c->L.masked, pattern(c),
                                      c->P, (float *)dr, (float *)du, (float *)dT, c->stream);
    if (e != cudaSuccess) return cuda_fail(c, e, "macroscopic kernel");
    return LBM_OK;
}

lbm_status lbm_diagnostics(lbm_ctx *c, lbm_diag *out)
{
    if (!c) return fail(nullptr, LBM_ERR_ARG, "ctx is NULL");
    if (!out) return fail(c, LBM_ERR_ARG, "out is NULL");
    if (c->cells_left) return partly_stepped(c);
    if (!c->initialized) return fail(c, LBM_ERR_STATE, "no state: call lbm_init_equilibrium");
    DeviceGuard guard(c->device);
    cudaError_t e = lbm::launch_diag(c->cfg.lattice, c->cfg.thermal, c->L.masked, pattern(c),
                                     c->P, c->partial, c->result, c->stream);
    if (e != cudaSuccess) return cuda_fail(c, e, "diagnostics kernel");
    double r[lbm::DIAG_N] = {0};
    e = cudaMemcpyAsync(r, c->result, sizeof(double) * lbm::DIAG_VALUES,
                        cudaMemcpyDeviceToHost, c->stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(c->stream);
    if (e != cudaSuccess) return cuda_fail(c, e, "diagnostics read-back");
    std::memset(out, 0, sizeof(*out));
    out->fluid_cells = (long long)std::llround(r[14]);
    out->mass = (double)out->fluid_cells + r[0];
    for (int a = 0; a < 3; ++a) {
        out->momentum[a] = r[1 + a];
        out->force[a] = r[4 + a];
    }
    for (int i = 0; i < 6; ++i) out->heat[i] = r[7 + i];
    out->steps = c->steps;
    out->finite = r[13] == 0.0 && std::isfinite(r[0]);
    // Nusselt numbers of the hottest and coldest Dirichlet faces
    const lbm::Params &P = c->P;
    int hot = -1, cold = -1;
    for (int i = 0; i < 6; ++i) {
        if (!P.face_dir[i]) continue;
        if (hot < 0 || c->cfg.T_wall[i] > c->cfg.T_wall[hot]) hot = i;
        if (cold < 0 || c->cfg.T_wall[i] < c->cfg.T_wall[cold]) cold = i;
    }
    if (hot >= 0 && cold >= 0 && c->cfg.T_wall[hot] > c->cfg.T_wall[cold]) {
        const double dT = c->cfg.T_wall[hot] - c->cfg.T_wall[cold];
        const int n[3] = {c->cfg.nx, c->cfg.ny, c->cfg.nz};
        auto nusselt = [&](int face) {
            const int a = face / 2;
            const double area = (double)n[0] * n[1] * n[2] / n[a];
            return std::fabs(out->heat[face]) * n[a] / (dT * area);
        };
        out->nu_hot = nusselt(hot);
        out->nu_cold = nusselt(cold);
        // volume average along the hot-cold axis: 1 + <u_a T> H / (kappa dT), with the
        // flux counted from the hot face towards the cold one
        const int a = hot / 2;
        if (cold / 2 == a && c->cfg.thermal && out->fluid_cells > 0) {
            const double omega = c->cfg.thermal == LBM_D2Q5 ? (4.0 + c->cfg.a_T) / 10.0
                                                            : (6.0 + c->cfg.a_T) / 21.0;
            const double kappa = omega * (1.0 / c->cfg.s_T[1 + a] - 0.5);
            const double sign = (hot % 2 == 0) ? 1.0 : -1.0;
            const double uT = r[15 + a] / (double)out->fluid_cells;
            out->nu_volume = 1.0 + sign * uT * n[a] / (kappa * dT);
        }
    }
    for (int a = 0; a < 3; ++a) out->uT[a] = r[15 + a];
    out->ib_samples = c->P.ib_n;
    if (c->P.ib_n > 0) {
        // reaction force and torque of the last step's penalties (fp64 on the host), over
        // the samples kept (dropped ones are ordered last)
        const size_t cap = c->L.ib_cap;
        std::vector<float> xs(8 * cap), gs(3 * cap);   // x3 ub3 w kept; g3
        unsigned dropped = 0;
        e = cudaMemcpyAsync(xs.data(), c->P.ibx, sizeof(float) * xs.size(),
                            cudaMemcpyDeviceToHost, c->stream);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(gs.data(), c->P.ibg, sizeof(float) * gs.size(),
                                cudaMemcpyDeviceToHost, c->stream);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(&dropped, lbm::ib_dropped_counter(c->P, c->ws + c->L.off_ibsort),
                                sizeof(unsigned), cudaMemcpyDeviceToHost, c->stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize(c->stream);
        if (e != cudaSuccess) return cuda_fail(c, e, "immersed-boundary read-back");
        out->ib_dropped = (int)dropped;
        // centroid of the kept samples (plane 7 flags them); dropped ones exert no force
        const int n = c->P.ib_n;
        double centre[3] = {0, 0, 0}, kept = 0.0;
        for (int s = 0; s < n; ++s) {
            if (xs[7 * cap + s] == 0.0f) continue;
            kept += 1.0;
            for (int a = 0; a < 3; ++a) centre[a] += (double)xs[a * cap + s];
        }
        for (int a = 0; a < 3; ++a) centre[a] = kept > 0 ? centre[a] / kept : 0.0;
        for (int s = 0; s < n; ++s) {
            if (xs[7 * cap + s] == 0.0f) continue;
            const double g[3] = {gs[s], gs[cap + s], gs[2 * cap + s]};
            const double r[3] = {xs[s] - centre[0], xs[cap + s] - centre[1],
                                 xs[2 * cap + s] - centre[2]};
            for (int a = 0; a < 3; ++a) out->ib_force[a] -= g[a];
            out->ib_torque[0] -= r[1] * g[2] - r[2] * g[1];
            out->ib_torque[1] -= r[2] * g[0] - r[0] * g[2];
            out->ib_torque[2] -= r[0] * g[1] - r[1] * g[0];
        }
    }
    if (!out->finite) return fail(c, LBM_ERR_NONFINITE, "non-finite rho or T in the state");
    return LBM_OK;
}

lbm_status lbm_solid_force(lbm_ctx *c, double F_out[3])
{
    if (!c) return fail(nullptr, LBM_ERR_ARG, "ctx is NULL");
    if (!F_out) return fail(c, LBM_ERR_ARG, "F_out is NULL");
    lbm_diag d;
    lbm_status s = lbm_diagnostics(c, &d);
    if (s != LBM_OK && s != LBM_ERR_NONFINITE) return s;
    for (int a = 0; a < 3; ++a) F_out[a] = d.force[a];
    return s;
}

static lbm_status populations(lbm_ctx *c, float *f, float *g, bool set)
{
    if (!c) return fail(nullptr, LBM_ERR_ARG, "ctx is NULL");
    if (c->cells_left) return partly_stepped(c);
    if (!f) return fail(c, LBM_ERR_ARG, "f is NULL");
    if (c->L.QT && !g && set) return fail(c, LBM_ERR_ARG, "g is required with a thermal lattice");
    if (!set && !c->initialized) return fail(c, LBM_ERR_STATE, "no state to read");
    DeviceGuard guard(c->device);
    void *df, *dg = nullptr;
    lbm_status s = device_address(c, f, "f", &df);
    if (s == LBM_OK && g && c->L.QT) s = device_address(c, g, "g", &dg);
    if (s != LBM_OK) return s;
    cudaError_t e = lbm::launch_pop(c->cfg.lattice, c->cfg.thermal, c->L.masked, pattern(c), set,
                                    c->P, (float *)df, (float *)dg, c->stream);
    if (e != cudaSuccess) return cuda_fail(c, e, set ? "set kernel" : "get kernel");
    if (set) {
        c->initialized = true;
        c->steps = 0;
    }
    return LBM_OK;
}

lbm_status lbm_get_populations(lbm_ctx *c, float *f, float *g)
{
    return populations(c, f, g, false);
}

lbm_status lbm_set_populations(lbm_ctx *c, const float *f, const float *g)
{
    return populations(c, const_cast<float *>(f), const_cast<float *>(g), true);
}

lbm_status lbm_get_link_mask(lbm_ctx *c, uint32_t *mask)
{
    if (!c) return fail(nullptr, LBM_ERR_ARG, "ctx is NULL");
    if (!mask) return fail(c, LBM_ERR_ARG, "mask is NULL");
    DeviceGuard guard(c->device);
    void *dm;
    lbm_status s = device_address(c, mask, "mask", &dm);
    if (s != LBM_OK) return s;
    cudaError_t e;
    if (c->L.masked)
        e = cudaMemcpyAsync(dm, c->P.mask, sizeof(uint32_t) * (size_t)c->L.N,
                            cudaMemcpyDefault, c->stream);
    else
        e = cudaMemsetAsync(dm, 0, sizeof(uint32_t) * (size_t)c->L.N, c->stream);
    if (e != cudaSuccess) return cuda_fail(c, e, "mask copy");
    return LBM_OK;
}

lbm_status lbm_set_ib_samples(lbm_ctx *c, int n, const float *xyz, const float *ub,
                              const float *weight)
{
    if (!c) return fail(nullptr, LBM_ERR_ARG, "ctx is NULL");
    if (c->L.ib_cap <= 0) return fail(c, LBM_ERR_STATE, "created with ib_max_samples = 0");
    if (n < 0 || n > c->L.ib_cap)
        return fail(c, LBM_ERR_ARG, "n must lie in [0, ib_max_samples]");
    if (n > 0 && !xyz) return fail(c, LBM_ERR_ARG, "xyz is required");
    DeviceGuard guard(c->device);
    const int dim = c->L.dim;
    const int ext[3] = {c->cfg.nx, c->cfg.ny, c->cfg.nz};
    const int l = c->cfg.ib_block > 0 ? c->cfg.ib_block : 4;
    // positions: wrap periodic axes, check wall axes
    std::vector<float> x(3 * (size_t)n);
    for (int s = 0; s < n; ++s) {
        float v[3];
        if (!lbm::ib_place(c->P, dim, xyz + 3 * s, v)) {
            for (int a = 0; a < dim; ++a)
                if (!std::isfinite(xyz[3 * s + a]))
                    return fail(c, LBM_ERR_ARG, "non-finite sample position");
            return fail(c, LBM_ERR_ARG,
                        "sample " + std::to_string(s) +
                            ": its stencil would leave the domain through a wall face");
        }
        for (int a = 0; a < 3; ++a) x[3 * s + a] = v[a];
    }
    // order: l x l x l blocks in x-y-z order, Morton code of the position inside a block
    const long long nbx = (ext[0] + l - 1) / l, nby = (ext[1] + l - 1) / l;
    std::vector<std::pair<unsigned long long, int>> key(n);
    for (int s = 0; s < n; ++s) {
        const float v[3] = {x[3 * s], x[3 * s + 1], x[3 * s + 2]};
        key[s] = {lbm::ib_sort_key(v, dim, l, nbx, nby), s};
    }
    std::stable_sort(key.begin(), key.end());
    const size_t cap = c->L.ib_cap;
    std::vector<float> host(8 * cap, 0.0f);   // planes: x, y, z, ub x3, w, kept
    std::vector<int> perm(std::max(n, 1));
    for (int i = 0; i < n; ++i) {
        const int s = key[i].second;
        perm[i] = s;
        for (int a = 0; a < 3; ++a) {
            host[a * cap + i] = x[3 * s + a];
            host[(3 + a) * cap + i] = (ub && a < dim) ? ub[3 * s + a] : 0.0f;
        }
        host[6 * cap + i] = weight ? weight[s] : 1.0f;
        host[7 * cap + i] = 1.0f;
    }
    uint32_t *mask = const_cast<uint32_t *>(c->P.mask);
    void *scratch = c->ws + c->L.off_ibsort;
    // clear the current samples' stencil marks before their positions are overwritten
    cudaError_t e = lbm::launch_ib_mark(c->cfg.lattice, c->P, mask, false, c->stream);
    if (e != cudaSuccess) return cuda_fail(c, e, "clearing the samples' stencils");
    e = cudaMemcpyAsync(const_cast<float *>(c->P.ibx), host.data(), sizeof(float) * host.size(),
                        cudaMemcpyHostToDevice, c->stream);
    // the order, for lbm_set_ib_samples_device calls that keep it
    if (e == cudaSuccess && n > 0)
        e = cudaMemcpyAsync(lbm::ib_order_perm(c->P, scratch), perm.data(), sizeof(int) * n,
                            cudaMemcpyHostToDevice, c->stream);
    if (e == cudaSuccess)
        e = cudaMemsetAsync(lbm::ib_dropped_counter(c->P, scratch), 0, sizeof(unsigned),
                            c->stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(c->stream);   // host buffer lifetime
    if (e != cudaSuccess) return cuda_fail(c, e, "copy of the samples");
    c->ib_order_n = n;
    c->P.ib_n = n;
    c->drop_graphs();   // captured steps hold the sample count
    e = lbm::launch_ib_mark(c->cfg.lattice, c->P, mask, true, c->stream);
    if (e != cudaSuccess) return cuda_fail(c, e, "marking the samples' stencils");
    return LBM_OK;
}

lbm_status lbm_set_ib_samples_device(lbm_ctx *c, int n, const float *xyz, const float *ub,
                                     const float *weight, int reorder)
{
    if (!c) return fail(nullptr, LBM_ERR_ARG, "ctx is NULL");
    if (c->L.ib_cap <= 0) return fail(c, LBM_ERR_STATE, "created with ib_max_samples = 0");
    if (n < 0 || n > c->L.ib_cap)
        return fail(c, LBM_ERR_ARG, "n must lie in [0, ib_max_samples]");
    if (n > 0 && !xyz) return fail(c, LBM_ERR_ARG, "xyz is required");
    if (!reorder && n != c->ib_order_n)
        return fail(c, LBM_ERR_STATE,
                    "no stored sample order for " + std::to_string(n) +
                        " samples: order them first (reorder != 0 or lbm_set_ib_samples)");
    DeviceGuard guard(c->device);
    void *dx = nullptr, *du = nullptr, *dw = nullptr;
    lbm_status st = LBM_OK;
    if (n > 0) st = device_address(c, xyz, "xyz", &dx);
    if (st == LBM_OK && n > 0 && ub) st = device_address(c, ub, "ub", &du);
    if (st == LBM_OK && n > 0 && weight) st = device_address(c, weight, "weight", &dw);
    if (st != LBM_OK) return st;
    const int l = c->cfg.ib_block > 0 ? c->cfg.ib_block : 4;
    uint32_t *mask = const_cast<uint32_t *>(c->P.mask);
    void *scratch = c->ws + c->L.off_ibsort;
    cudaError_t e = lbm::launch_ib_mark(c->cfg.lattice, c->P, mask, false, c->stream);
    if (e != cudaSuccess) return cuda_fail(c, e, "clearing the samples' stencils");
    if (n > 0) {
        e = lbm::launch_ib_order(c->cfg.lattice, c->P, n, l, static_cast<const float *>(dx),
                                 static_cast<const float *>(du), static_cast<const float *>(dw),
                                 scratch, reorder != 0, c->stream);
    } else {
        e = cudaMemsetAsync(lbm::ib_dropped_counter(c->P, scratch), 0, sizeof(unsigned),
                            c->stream);
    }
    if (e != cudaSuccess) return cuda_fail(c, e, "ordering the samples");
    c->ib_order_n = n;
    if (c->P.ib_n != n) c->drop_graphs();   // captured steps hold the sample count
    c->P.ib_n = n;
    e = lbm::launch_ib_mark(c->cfg.lattice, c->P, mask, true, c->stream);
    if (e != cudaSuccess) return cuda_fail(c, e, "marking the samples' stencils");
    return LBM_OK;
}

namespace {

// Populations per plane cell that cross a face (momentum + thermal), on any axis.
int halo_directions(const lbm_ctx *c)
{
    const int thermal = c->L.QT ? 1 : 0;
    if (c->cfg.lattice == LBM_D3Q27) return 9;        // every c with c_axis = +-1
    return c->cfg.lattice == LBM_D3Q19 ? 5 + thermal : 3 + thermal;
}

size_t halo_plane_cells(const lbm_ctx *c, int axis)
{
    const size_t n[3] = {(size_t)c->cfg.nx, (size_t)c->cfg.ny, (size_t)c->cfg.nz};
    return n[axis == 0 ? 1 : 0] * n[axis == 2 ? 1 : 2];
}

lbm_status halo_call(lbm_ctx *c, int axis, int side, int phase, int unpack, const void *buf)
{
    if (!c) return fail(nullptr, LBM_ERR_ARG, "ctx is NULL");
    if (!c->L.halo) return fail(c, LBM_ERR_STATE, "no HALO face in this context");
    if (axis < 0 || axis >= c->L.dim) return fail(c, LBM_ERR_ARG, "axis out of range");
    if (side != 0 && side != 1) return fail(c, LBM_ERR_ARG, "side must be 0 (low) or 1 (high)");
    const int face = 2 * axis + side;
    if (c->cfg.face_flow[face] != LBM_FACE_HALO)
        return fail(c, LBM_ERR_ARG, "that side is not a HALO face");
    if (phase != LBM_HALO_FILL && phase != LBM_HALO_DRAIN)
        return fail(c, LBM_ERR_ARG, "phase must be LBM_HALO_FILL or LBM_HALO_DRAIN");
    if (!c->initialized) return fail(c, LBM_ERR_STATE, "no state");
    if (phase == LBM_HALO_FILL && c->parity != 1)
        return fail(c, LBM_ERR_STATE, "FILL belongs before an odd step (parity 1)");
    if (phase == LBM_HALO_DRAIN && (c->parity != 0 || c->steps == 0))
        return fail(c, LBM_ERR_STATE, "DRAIN belongs after an odd step (parity 0)");
    if (!buf) return fail(c, LBM_ERR_ARG, "buf is NULL");
    DeviceGuard guard(c->device);
    void *db;
    lbm_status st = device_address(c, buf, "buf", &db);
    if (st != LBM_OK) return st;
    cudaError_t e = lbm::launch_halo(c->cfg.lattice, c->cfg.thermal, c->P, axis, side, phase,
                                     unpack, static_cast<float *>(db), c->stream);
    if (e != cudaSuccess) return cuda_fail(c, e, "halo kernel");
    return LBM_OK;
}

}  // namespace

lbm_status lbm_halo_bytes(const lbm_ctx *c, size_t *bytes)
{
    if (!c || !bytes) return fail(nullptr, LBM_ERR_ARG, "ctx and bytes are required");
    *bytes = c->L.halo ? sizeof(float) * halo_directions(c) * halo_plane_cells(c, c->L.dim - 1)
                       : 0;
    return LBM_OK;
}

lbm_status lbm_halo_pack(lbm_ctx *c, int side, int phase, void *buf)
{
    return halo_call(c, c ? c->L.dim - 1 : 0, side, phase, 0, buf);
}

lbm_status lbm_halo_unpack(lbm_ctx *c, int side, int phase, const void *buf)
{
    return halo_call(c, c ? c->L.dim - 1 : 0, side, phase, 1, buf);
}

lbm_status lbm_halo_axis_bytes(const lbm_ctx *c, int axis, size_t *bytes)
{
    if (!c || !bytes) return fail(nullptr, LBM_ERR_ARG, "ctx and bytes are required");
    if (axis < 0 || axis >= c->L.dim)
        return fail(const_cast<lbm_ctx *>(c), LBM_ERR_ARG, "axis out of range");
    *bytes = c->L.halo ? sizeof(float) * halo_directions(c) * halo_plane_cells(c, axis) : 0;
    return LBM_OK;
}

lbm_status lbm_halo_axis_pack(lbm_ctx *c, int axis, int side, int phase, void *buf)
{
    return halo_call(c, axis, side, phase, 0, buf);
}

lbm_status lbm_halo_axis_unpack(lbm_ctx *c, int axis, int side, int phase, const void *buf)
{
    return halo_call(c, axis, side, phase, 1, buf);
}

namespace {

// The checks of one face swap (lbm_halo_axis_swap); errors are recorded on lo.
lbm_status check_swap(lbm_ctx *lo, lbm_ctx *hi, int axis, int phase)
{
    if (!lo || !hi) return fail(nullptr, LBM_ERR_ARG, "both contexts are required");
    if (!lo->L.halo || !hi->L.halo) return fail(lo, LBM_ERR_STATE, "no HALO face in a context");
    if (axis < 0 || axis >= lo->L.dim) return fail(lo, LBM_ERR_ARG, "axis out of range");
    if (lo->cfg.face_flow[2 * axis + 1] != LBM_FACE_HALO ||
        hi->cfg.face_flow[2 * axis] != LBM_FACE_HALO)
        return fail(lo, LBM_ERR_ARG, "lo's high face and hi's low face must be HALO faces");
    if (phase != LBM_HALO_FILL && phase != LBM_HALO_DRAIN)
        return fail(lo, LBM_ERR_ARG, "phase must be LBM_HALO_FILL or LBM_HALO_DRAIN");
    if (lo->cfg.lattice != hi->cfg.lattice || lo->cfg.thermal != hi->cfg.thermal)
        return fail(lo, LBM_ERR_ARG, "the two contexts must have the same lattices");
    const int nlo[3] = {lo->cfg.nx, lo->cfg.ny, lo->cfg.nz};
    const int nhi[3] = {hi->cfg.nx, hi->cfg.ny, hi->cfg.nz};
    for (int a = 0; a < 3; ++a)
        if (a != axis && nlo[a] != nhi[a])
            return fail(lo, LBM_ERR_ARG, "the two faces must have the same extents");
    if (lo->device != hi->device)
        return fail(lo, LBM_ERR_UNSUPPORTED, "the two contexts must be on one device");
    if (!lo->initialized || !hi->initialized) return fail(lo, LBM_ERR_STATE, "no state");
    if (lo->parity != hi->parity || lo->steps != hi->steps)
        return fail(lo, LBM_ERR_STATE, "the two contexts must be at the same step");
    if (phase == LBM_HALO_FILL && lo->parity != 1)
        return fail(lo, LBM_ERR_STATE, "FILL belongs before an odd step (parity 1)");
    if (phase == LBM_HALO_DRAIN && (lo->parity != 0 || lo->steps == 0))
        return fail(lo, LBM_ERR_STATE, "DRAIN belongs after an odd step (parity 0)");
    return LBM_OK;
}

}  // namespace

lbm_status lbm_halo_axis_swap(lbm_ctx *lo, lbm_ctx *hi, int axis, int phase)
{
    lbm_status st = check_swap(lo, hi, axis, phase);
    if (st != LBM_OK) return st;
    DeviceGuard guard(lo->device);
    cudaError_t e = lbm::launch_halo_swap(lo->cfg.lattice, lo->cfg.thermal, lo->P, hi->P, axis,
                                          phase, lo->stream);
    if (e != cudaSuccess) return cuda_fail(lo, e, "halo swap kernel");
    return LBM_OK;
}

lbm_status lbm_halo_axis_swap_many(lbm_ctx *const *lo, lbm_ctx *const *hi, int n, int axis,
                                   int phase)
{
    if (!lo || !hi) return fail(nullptr, LBM_ERR_ARG, "lo and hi are required");
    if (n < 1 || n > lbm::HALO_MAX_PAIRS)
        return fail(nullptr, LBM_ERR_ARG,
                    "n must lie in [1, " + std::to_string(lbm::HALO_MAX_PAIRS) + "]");
    lbm::HaloPairs pairs{};
    pairs.n = n;
    for (int p = 0; p < n; ++p) {
        lbm_status st = check_swap(lo[p], hi[p], axis, phase);
        if (st != LBM_OK) {
            if (p > 0 && lo[p] && lo[0]) lo[0]->err = lo[p]->err;   // the call's error on lo[0]
            return st;
        }
        if (lo[p]->device != lo[0]->device || lo[p]->cfg.lattice != lo[0]->cfg.lattice ||
            lo[p]->cfg.thermal != lo[0]->cfg.thermal || lo[p]->parity != lo[0]->parity ||
            lo[p]->steps != lo[0]->steps)
            return fail(lo[0], LBM_ERR_ARG,
                        "every pair must be on one device, with the same lattices, at one step");
        // each face once: no context may be `lo` (or `hi`) of two pairs
        for (int q = 0; q < p; ++q)
            if (lo[q] == lo[p] || hi[q] == hi[p])
                return fail(lo[0], LBM_ERR_ARG, "a face appears in two pairs");
        pairs.lo[p].from_params(lo[p]->P);
        pairs.hi[p].from_params(hi[p]->P);
    }
    DeviceGuard guard(lo[0]->device);
    cudaError_t e = lbm::launch_halo_swap_many(lo[0]->cfg.lattice, lo[0]->cfg.thermal, pairs,
                                               axis, phase, lo[0]->stream);
    if (e != cudaSuccess) return cuda_fail(lo[0], e, "halo swap kernel (pairs)");
    return LBM_OK;
}

lbm_status lbm_set_stream(lbm_ctx *c, void *cuda_stream)
{
    if (!c) return fail(nullptr, LBM_ERR_ARG, "ctx is NULL");
    c->stream = static_cast<cudaStream_t>(cuda_stream);
    return LBM_OK;
}

int lbm_parity(const lbm_ctx *c) { return c ? c->parity : -1; }

long long lbm_steps_taken(const lbm_ctx *c) { return c ? c->steps : -1; }

const char *lbm_last_error(const lbm_ctx *c) { return c ? c->err.c_str() : g_error.c_str(); }

const char *lbm_version(void) { return "lbm-gb300 0.1 (sm_103a, AA in-place, fp32)"; }

void lbm_destroy(lbm_ctx *c) { delete c; }

}  // extern "C"
