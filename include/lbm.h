/*
 * lbm.h -- C ABI of the GB300 (sm_103a) lattice-Boltzmann collide-and-stream library.
 *
 * One library call advances a lattice-Boltzmann flow (D3Q19 or D2Q9 populations with BGK
 * or MRT collision, or D3Q27 populations with central-moment MRT; Guo forcing with
 * Boussinesq buoyancy; optional D3Q7 / D2Q5 thermal populations) by n time steps, one fused kernel launch per step, populations streamed in
 * place with the AA pattern in a single fp32 structure-of-arrays buffer.
 *
 * Sources (the method each call implements):
 *   [TLBM] "Multi-GPU thermal lattice Boltzmann simulations using OpenACC and MPI",
 *          Sec. 2: Eq. 5 (MRT evolution of f, forcing F' = M^-1 (I - S/2) M F~),
 *          rho = sum f_i, u = (sum e_i f_i + F/2) / rho, F = rho g beta_T (T - T0) along
 *          the vertical axis, half-way bounce-back f_ibar(x, t+1) = f_i+(x, t); Eq. 7
 *          (MRT evolution of g), T = sum g_i, half-way anti-bounce-back
 *          g_ibar(x, t+1) = -g_i+(x, t) + omega T_w with omega = (4 + a_T)/10 (D2Q5) or
 *          (6 + a_T)/21 (D3Q7), adiabatic walls by half-way bounce-back;
 *          Sec. 3: SoA index x + Nx y + Nx Ny z + Nx Ny Nz i; the MLUPS metric.
 *   [AA]   "GPU lattice Boltzmann: streaming layout and performance": the in-place AA
 *          pattern (even steps read (q, x) and write (opposite(q), x); odd steps read
 *          (opposite(q), x - c_q) and write (q, x + c_q)), 152 bytes per D3Q19 update,
 *          momentum exchange read back from the last step of a submission.
 *   [KFS]  "GPU Optimization for High-Quality Kinetic Fluid Simulation", Sec. 3.1,
 *          Eq. 1-5 (lattice Boltzmann equation, moments, pull streaming, MRT collision
 *          Omega = -M^-1 D (m - m_eq)); Fig. 2 (the D3Q27 lattice, central moments);
 *          Sec. 4 (SoA layout, bounce-back at solid nodes).
 *
 * Conventions shared by every call:
 *   - Memory.  The caller owns all device memory: it allocates one device workspace of
 *     lbm_workspace_bytes() bytes and passes it to lbm_create(); the library carves the
 *     populations, the link mask and the reduction scratch out of it and never calls
 *     cudaMalloc or cudaFree.  The library owns only the small host-side context.
 *   - Fields.  fp32, structure of arrays, x fastest: a scalar field is nx*ny*nz floats
 *     (index x + nx*(y + ny*z)); the velocity is dim such planes, component-major
 *     (u_x plane, then u_y, then u_z in 3-D).  Populations in get/set are Q planes
 *     (q-major) of nx*ny*nz floats, in the lattice order given below.  Solid cells read
 *     out as rho = u = T = 0 and populations 0.
 *   - Field pointers may be device memory or page-locked host memory (cudaHostAlloc /
 *     cudaHostRegister; the kernel then reads or writes it over the host link).  Pageable
 *     host memory is accepted only where the device reports pageable-memory access.
 *   - Ordering.  All device work is enqueued on the stream given to lbm_create(), in call
 *     order, and returns without waiting, except lbm_solid_force() and lbm_diagnostics(),
 *     which wait for that stream.
 *   - Errors.  Every call returns an lbm_status.  Argument errors are found on the host
 *     before anything is enqueued.  A CUDA error is returned as LBM_ERR_CUDA; its text is
 *     available from lbm_last_error().  No call aborts, traps or throws across the ABI.
 *
 * Lattice orders (c_q):
 *   D3Q19: 0 rest; 1 +x, 2 -x, 3 +y, 4 -y, 5 +z, 6 -z; 7 (+,+,0), 8 (-,+,0), 9 (+,-,0),
 *          10 (-,-,0); 11 (+,0,+), 12 (-,0,+), 13 (+,0,-), 14 (-,0,-); 15 (0,+,+),
 *          16 (0,-,+), 17 (0,+,-), 18 (0,-,-).
 *   D3Q27: 0-18 as D3Q19; 19 (+,+,+), 20 (-,+,+), 21 (+,-,+), 22 (-,-,+), 23 (+,+,-),
 *          24 (-,+,-), 25 (+,-,-), 26 (-,-,-).
 *   D2Q9:  0 rest; 1 +x, 2 +y, 3 -x, 4 -y, 5 (+,+), 6 (-,+), 7 (-,-), 8 (+,-).
 *   D3Q7:  0 rest; 1 +x, 2 -x, 3 +y, 4 -y, 5 +z, 6 -z.   D2Q5: 0 rest; 1 +x, 2 +y, 3 -x, 4 -y.
 * Moment rows (index of s[] / s_T[]):
 *   D3Q19 (d'Humieres basis): 0 rho, 1 e, 2 eps, 3 jx, 4 qx, 5 jy, 6 qy, 7 jz, 8 qz,
 *          9 3pxx, 10 3pixx, 11 pww, 12 piww, 13 pxy, 14 pyz, 15 pxz, 16 mx, 17 my, 18 mz.
 *   D2Q9 (Lallemand-Luo basis): 0 rho, 1 e, 2 eps, 3 jx, 4 qx, 5 jy, 6 qy, 7 pxx, 8 pxy.
 *   D3Q7: 0 T, 1-3 jx..jz, 4 e (rest weight -6), 5 (0,2,2,-1,-1,-1,-1), 6 (0,0,0,1,1,-1,-1).
 *   D2Q5: 0 T, 1 jx, 2 jy, 3 e (rest weight -4), 4 (0,1,-1,1,-1).
 *   Rates of conserved rows (rho, j; T) are ignored.  Viscosity nu = (1/s_nu - 1/2)/3 on
 *   the stress rows; thermal diffusivity kappa = omega (1/s_kappa - 1/2) on the j rows.
 *   D3Q27 central moments (LBM_CM): the 27 moments prod_a (c_a - u_a)^e_a, e in {0,1,2}^3,
 *          about u = (j + F/2)/rho, with the second-order normal ones taken as xx - yy,
 *          xx - zz (shear rate 1/tau, like xy, xz, yz; nu = (tau - 1/2)/3) and xx + yy + zz
 *          (rate cm_rates[0]); orders 3, 4, 5, 6 relax at cm_rates[1..4]; orders 0, 1 are
 *          conserved.  Equilibrium central moments rho prod_a (1, 0, 1/3)[e_a] (discrete
 *          form: the product rho prod_a phi(c_a, u_a), phi(0, u) = 2/3 - u^2,
 *          phi(+-1, u) = (1/3 + u^2 +- u)/2, also the initial state); the force enters as
 *          the central moments of (F/rho) . d f_eq / du, relaxed with (I - D/2).
 */
#ifndef LBM_GB300_H
#define LBM_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct lbm_ctx lbm_ctx; /* opaque, host side */

typedef enum {
    LBM_OK = 0,
    LBM_ERR_ARG = 1,         /* bad argument (null pointer, size, range)            */
    LBM_ERR_UNSUPPORTED = 2, /* valid but not supported combination                 */
    LBM_ERR_WORKSPACE = 3,   /* workspace missing, too small or misaligned          */
    LBM_ERR_CUDA = 4,        /* a CUDA runtime call or kernel launch failed         */
    LBM_ERR_NONFINITE = 5,   /* diagnostics found a non-finite rho or T             */
    LBM_ERR_STATE = 6        /* call out of order (e.g. stepping before any init)   */
} lbm_status;

enum { LBM_D2Q9 = 9, LBM_D3Q19 = 19, LBM_D3Q27 = 27 };
enum { LBM_THERMAL_NONE = 0, LBM_D2Q5 = 5, LBM_D3Q7 = 7 };
/* LBM_CM: central-moment MRT, D3Q27 only (and the only collision of D3Q27) */
enum { LBM_BGK = 0, LBM_MRT = 1, LBM_CM = 2 };
enum { LBM_FACE_PERIODIC = 0, LBM_FACE_WALL = 1 };        /* flow: half-way bounce-back */
/* A slab face: the context is one slab of a larger domain, split along its outer axis (z
 * in 3-D, y in 2-D), or one block of a domain split along several axes.  The grid then
 * includes one ghost plane at each HALO face (the first / last plane of that axis); ghost
 * cells are never updated and hold the neighbouring slab's or block's populations, moved by
 * lbm_halo_pack / lbm_halo_unpack and their per-axis forms ([TLBM] Sec. 3). */
enum { LBM_FACE_HALO = 2 };
enum { LBM_HALO_FILL = 0, LBM_HALO_DRAIN = 1 };
enum { LBM_TFACE_ADIABATIC = 0, LBM_TFACE_DIRICHLET = 1 }; /* thermal, on WALL faces   */
/* Population layout ([AA] Options::streaming): AA = one buffer streamed in place (152 B
 * per D3Q19 update); PULL = two buffers, one fused pull-collide kernel per step (152 B,
 * twice the memory); SPLIT = two buffers, collide in place then pull into the other
 * buffer, two kernels per step (304 B). */
enum { LBM_STREAM_AA = 0, LBM_STREAM_PULL = 1, LBM_STREAM_SPLIT = 2 };

/* Problem description ([TLBM] Sec. 2; [KFS] Sec. 3.1).  Face order: -x, +x, -y, +y, -z, +z.
 * Both faces of an axis must have the same flow kind.  A link is a wall link when its
 * far end lies outside the domain through a WALL face or is a solid cell; wall links
 * bounce back f, and bounce back g (adiabatic face or solid) or anti-bounce-back g
 * (DIRICHLET face, wall temperature T_wall[face]). */
typedef struct {
    int nx, ny, nz;       /* cells; nz == 1 for D2Q9; nx*ny*nz < 2^31; nz <= 65535;
                             ny <= 65535 (131070 when nx <= 32): launch-grid extents     */
    int lattice;          /* LBM_D3Q19, LBM_D2Q9 or LBM_D3Q27                          */
    int thermal;          /* LBM_THERMAL_NONE, LBM_D3Q7 (with D3Q19), LBM_D2Q5 (D2Q9)  */
    int collision;        /* LBM_BGK or LBM_MRT (D3Q19, D2Q9); LBM_CM (D3Q27)           */
    double tau;           /* BGK relaxation time, > 1/2; LBM_CM: 1/tau = shear rate    */
    double s[19];         /* MRT rate of each moment row, in [0, 2)                    */
    double s_T[7];        /* thermal MRT rate of each row, in [0, 2)                   */
    double cm_rates[5];   /* LBM_CM: bulk rate, then orders 3, 4, 5, 6; each in (0, 2).
                             D3Q27 takes no thermal lattice and only LBM_STREAM_AA
                             (LBM_ERR_UNSUPPORTED).                                    */
    double a_T;           /* thermal energy-moment constant (e_eq = a_T T), in (-Q_T+1, 1) */
    double g_body[3];     /* body acceleration: F += rho g_body                        */
    double gbeta, T0;     /* buoyancy: F += rho gbeta (T - T0) e_up (thermal only)      */
    int up_axis;          /* 0, 1, 2 = x, y, z (2-D: 0 or 1)                           */
    int face_flow[6];     /* LBM_FACE_PERIODIC or LBM_FACE_WALL                        */
    int face_T[6];        /* LBM_TFACE_ADIABATIC or LBM_TFACE_DIRICHLET (WALL faces)    */
    double T_wall[6];     /* wall temperature of DIRICHLET faces                       */
    const uint8_t *solid_mask; /* HOST pointer, nx*ny*nz bytes, x fastest, nonzero =
                                  solid; NULL = no solid cells.  Read once by
                                  lbm_workspace_bytes and lbm_create (the bounding box
                                  of the solid cells, outside which the step derives
                                  the link mask from the coordinates) and copied by
                                  lbm_create; not kept. */
    int streaming;        /* LBM_STREAM_AA (default 0), LBM_STREAM_PULL or LBM_STREAM_SPLIT */
    int ib_max_samples;   /* capacity for immersed-boundary samples (0 = none); see
                             lbm_set_ib_samples                                          */
    int ib_block;         /* edge l (cells) of the blocks samples are ordered by; 0 = 4    */
} lbm_config;

/* Diagnostics of the current state (see lbm_diagnostics). */
typedef struct {
    double mass;          /* sum over fluid cells of rho                                  */
    double momentum[3];   /* sum over fluid cells of sum_q c_q f_q (no force shift)        */
    double force[3];      /* momentum exchanged with solid cells in the last step          */
    double heat[6];       /* per face: sum over fluid cells next to a DIRICHLET face of
                             2 (T_w - T), the wall-normal gradient over the half cell     */
    double nu_hot;        /* Nusselt number of the hottest / coldest DIRICHLET face:       */
    double nu_cold;       /*   |heat| * H / (dT * A), H = cells across, A = face cells     */
    long long fluid_cells;
    long long steps;      /* time steps taken since the last init / set                   */
    int finite;           /* 1 if every fluid rho (and T) is finite                        */
    int ib_samples;       /* immersed-boundary samples in use                              */
    double ib_force[3];   /* their reaction force -sum g_s in the last step               */
    double ib_torque[3];  /* -sum (x_s - centroid) x g_s about the samples' centroid      */
    double uT[3];         /* sum over fluid cells of u_a T, u = (j + F/2)/rho (thermal)    */
    double nu_volume;     /* volume-averaged Nusselt number along the axis of the hottest
                             and coldest DIRICHLET faces (when they face each other):
                             1 + <u_a T> H / (kappa dT), <.> over fluid cells, H = cells
                             across, kappa = omega (1/s_T[1 + a] - 1/2), the flux counted
                             from the hot face towards the cold one                      */
    int ib_dropped;       /* samples the last lbm_set_ib_samples_device dropped (invalid
                             positions); 0 after lbm_set_ib_samples                         */
} lbm_diag;

/* Bytes of device workspace lbm_create() needs for this configuration (validates it). */
lbm_status lbm_workspace_bytes(const lbm_config *cfg, size_t *bytes);

/* Validate cfg, carve the workspace (device memory, >= lbm_workspace_bytes bytes,
 * 256-byte aligned), copy the solid mask and build the per-cell link mask on
 * cuda_stream (a cudaStream_t; NULL = the legacy default stream).  *out receives the
 * context.  The context holds no state until lbm_init_equilibrium or lbm_set_populations. */
lbm_status lbm_create(const lbm_config *cfg, void *d_workspace, size_t workspace_bytes,
                      void *cuda_stream, lbm_ctx **out);

/* f = f_eq(rho, u) ([KFS] Eq. 2 inverted by the quadratic equilibrium), g = g_eq(T, u)
 * (equilibrium moments T, u T, a_T T, 0...), at every fluid cell; resets parity and the
 * step count.  rho: N floats, u: dim*N, T: N (NULL allowed only without thermal).  u is
 * used as given (no F/2 shift). */
lbm_status lbm_init_equilibrium(lbm_ctx *ctx, const float *rho, const float *u, const float *T);

/* Advance n >= 0 time steps ([TLBM] Eq. 5 and Eq. 7 fused with streaming, [AA]): one
 * kernel launch per step, alternating the even and odd AA forms (plus one immersed-boundary
 * launch per step when samples are set).  On grids of two or more waves of thread blocks
 * the step kernels are launched with programmatic stream serialization: a step's blocks may
 * be scheduled while the kernel before it on the stream is finishing, but they wait for
 * that kernel to complete, with its writes visible, before touching memory.  Work the
 * caller puts on the stream before or after lbm_step is therefore ordered as usual.  Grids
 * of at most 4 M cells replay captured graphs of 64 steps. */
lbm_status lbm_step(lbm_ctx *ctx, int n);

/* One time step split across calls by boxes of cells: each call launches the current step
 * (the same even or odd AA form lbm_step would launch) on the cells [lo, hi) only, lo and
 * hi host arrays of 3 ints (x, y, z; in 2-D lo[2] = 0, hi[2] = 1).  The step is complete,
 * and the parity and step count advance, once the calls since the last complete step have
 * covered every cell exactly once, in any order and any grouping; ghost cells of a slab or
 * block may be included, they are skipped.  The result is bit for bit that of lbm_step(1):
 * even steps only touch their own cells, and in the odd step every slot is read and then
 * written by one cell alone.  This lets a slab or block driver overlap its halo exchange
 * with the interior cells ([TLBM] Sec. 4, overlapping communication with computation; see
 * the halo calls below).  While a step is partly done, lbm_step, lbm_init_equilibrium,
 * lbm_macroscopic, lbm_diagnostics, lbm_solid_force and the population calls return
 * LBM_ERR_STATE; the halo calls are allowed.  Each call is one launch on the context's
 * stream, not chained to the work before it.  Errors: LBM_ERR_ARG for an empty box, a box
 * outside the grid, or one that overlaps a box already stepped in this step;
 * LBM_ERR_UNSUPPORTED for the two-buffer layouts and for contexts with immersed-boundary
 * capacity. */
lbm_status lbm_step_box(lbm_ctx *ctx, const int *lo, const int *hi);

/* lbm_step_box over the whole outer-axis planes [lo, hi) (z in 3-D, y in 2-D). */
lbm_status lbm_step_planes(lbm_ctx *ctx, int lo, int hi);

/* rho = sum f, u = (sum c f + F/2)/rho, T = sum g of the current state ([TLBM] Sec. 2).
 * Any of the three pointers may be NULL to skip that field. */
lbm_status lbm_macroscopic(lbm_ctx *ctx, float *rho, float *u, float *T);

/* Momentum exchanged with solid cells in the last step taken: the sum over links from a
 * fluid cell x into a solid cell of 2 f_q+(x) c_q ([AA]: read back from the step whose
 * forces are wanted).  Domain-face walls are not included.  Waits for the stream. */
lbm_status lbm_solid_force(lbm_ctx *ctx, double F_out[3]);

/* Mass, momentum, solid force, wall heat flux and Nusselt numbers, fp64 reductions.
 * Waits for the stream.  Returns LBM_ERR_NONFINITE (with *out filled) if a fluid rho or
 * T is not finite. */
lbm_status lbm_diagnostics(lbm_ctx *ctx, lbm_diag *out);

/* Copy the logical populations (parity resolved, f unshifted) out to / in from Q planes
 * (q-major, N floats each).  g may be NULL without a thermal lattice.  set resets the
 * step count but keeps the parity; get of a solid cell yields 0. */
lbm_status lbm_get_populations(lbm_ctx *ctx, float *f, float *g);
lbm_status lbm_set_populations(lbm_ctx *ctx, const float *f, const float *g);

/* Copy the per-cell link mask (N uint32): bit q (1..Q-1) = link q is a wall link,
 * bit 19+k (k = 1..Q_T-1) = thermal link k ends on a DIRICHLET face, bit 29 = ghost plane
 * of a slab, bit 30 = cell in an immersed-boundary sample's stencil, bit 31 = solid cell.
 * A context with no WALL face, solid mask or sample capacity keeps no mask and yields all
 * zeros (its ghost planes, if any, are known by their coordinate).  Device or page-locked
 * host destination. */
lbm_status lbm_get_link_mask(lbm_ctx *ctx, uint32_t *mask);

/* Immersed boundary ([KFS] Sec. 3.1, Eq. 6-8; sample order of its Sec. 4, Fig. 7).
 * Replace the solid samples: n <= cfg.ib_max_samples points xyz (HOST, 3n floats, cell
 * units: cell centres at integer coordinates), boundary velocities ub (HOST, 3n, NULL = 0)
 * and weights (HOST, n, NULL = 1).  Each later step, before the collision, interpolates
 * rho and u = (j + F_body/2)/rho at every sample from its 2x2x2 (2x2 in 2-D) stencil with
 * the trilinear kernel (Eq. 6), forms the penalty g = w rho (u_b - u) (Eq. 7) and
 * scatters it with the same kernel (Eq. 8, one thread per sample, atomic additions) into
 * a per-cell force added to that step's collision.  Solid stencil cells count as rho = 1,
 * u = 0 and take no force.  Positions on periodic axes are wrapped into the domain; on
 * wall axes they must satisfy 0 <= x < n - 1 so that the stencil stays inside
 * (LBM_ERR_ARG otherwise).  Samples are stored sorted by l x l x l block (x fastest) and
 * by Morton code inside a block, so that one warp's samples touch nearby cells.  n = 0
 * removes the boundary.  Enqueued on the context's stream; the host arrays may be freed on
 * return. */
lbm_status lbm_set_ib_samples(lbm_ctx *ctx, int n, const float *xyz, const float *ub,
                              const float *weight);

/* The same replacement with the samples in device memory (or page-locked host memory),
 * placed and ordered on the device: a body that moves every step updates its samples
 * without a host round trip.  Nothing waits for the stream; the arrays must stay valid
 * until the stream has run the call's kernels.
 *   reorder != 0: sort the samples ([KFS] Sec. 4: l-blocks, Morton code inside a block; the
 *     same order lbm_set_ib_samples gives) with a stable radix sort over (l-block, Morton)
 *     keys -- one thread block for up to 16384 samples, a multi-block pass per 8-bit digit
 *     beyond that -- and store the order;
 *   reorder == 0: place caller sample perm[i] in slot i, perm being the stored order of the
 *     last sort (of this call or of lbm_set_ib_samples), which must have had the same n
 *     (LBM_ERR_STATE otherwise).  A rigid body whose samples keep their indices keeps the
 *     locality of that sort while it moves, at the cost of one gather instead of a sort.
 * Placement is checked on the device: periodic axes wrap, and a sample with a non-finite
 * position or a stencil that would leave through a wall face is dropped -- it takes weight
 * 0 and position 0, is left out of the torque's centroid, and is counted in
 * lbm_diag.ib_dropped -- instead of failing the call.  Uses workspace that
 * lbm_workspace_bytes reserves with ib_max_samples. */
lbm_status lbm_set_ib_samples_device(lbm_ctx *ctx, int n, const float *xyz, const float *ub,
                                     const float *weight, int reorder);

/* Slab halos ([TLBM] Sec. 3: direction-selective exchange of contiguous buffers).  With
 * the AA pattern only odd steps read or write across a slab face, so a slab driver runs one
 * exchange after every lbm_step(1) of all its slabs:
 *   after an even step (parity now 1), FILL: for each HALO side s, lbm_halo_pack(s, FILL)
 *     here -> buffer -> the neighbour's lbm_halo_unpack(opposite s, FILL).  This supplies
 *     the ghost slots that the boundary cells read in the odd step, and from which their
 *     logical state is read (lbm_macroscopic, lbm_diagnostics ...) while the parity is 1;
 *   after an odd step (parity now 0), DRAIN: the same with phase DRAIN, returning what the
 *     boundary cells wrote into the ghost plane.  A DRAIN leaves alone a slot whose cell
 *     bounced that population back itself (the link towards the ghost is a wall link).
 * Between steps every owned cell then holds exactly what one undivided domain would hold.
 * Only the populations that cross the face move: 5 of 19 (D3Q19) + 1 of 7 (D3Q7), 3 of 9
 * (D2Q9) + 1 of 5 (D2Q5), per plane cell.
 *   side: 0 = low face of the outer axis, 1 = high face; it must be a HALO face.
 *   buf: device (or page-locked host) memory of lbm_halo_bytes bytes; packed as
 *        [direction][plane cell] fp32, momentum then thermal, directions in index order.
 * FILL is allowed at parity 1, DRAIN at parity 0 after at least one step (LBM_ERR_STATE
 * otherwise).  HALO faces need the AA layout and no immersed-boundary capacity
 * (LBM_ERR_UNSUPPORTED at create).  Stream-ordered; nothing waits.
 * Overlap with lbm_step_planes.  Call the planes next to a HALO face -- its ghost plane and
 * the first owned plane -- the boundary planes, the others the interior.  A pack reads
 * slots of the boundary planes (FILL: slots the even step wrote and the odd step leaves
 * alone; DRAIN: ghost slots the odd step wrote), and an unpack writes slots that only the
 * boundary planes' next step reads (FILL: ghost slots; DRAIN: slots the even step reads at
 * the first owned plane).  So, with the halo calls on a second stream (lbm_set_stream),
 * each step can run as: interior planes; wait for the previous exchange's unpack; boundary
 * planes; then this step's exchange, which overlaps the next step's interior planes.
 * lbm_halo_bytes gives 0 for a context without HALO faces. */
lbm_status lbm_halo_bytes(const lbm_ctx *ctx, size_t *bytes);
lbm_status lbm_halo_pack(lbm_ctx *ctx, int side, int phase, void *buf);
lbm_status lbm_halo_unpack(lbm_ctx *ctx, int side, int phase, const void *buf);

/* Block halos: the same exchange along any axis, for a domain split along several axes
 * (the multi-dimensional partitioning that [TLBM] Sec. 3 compares with slabs).  A context
 * may have HALO faces on every axis (x, y and z in 3-D; x and y in 2-D); its ghost planes
 * are then the first / last plane of each such axis, and the cells where ghost planes of
 * two or three axes meet are ghost cells too.  lbm_halo_axis_pack / _unpack move the plane
 * of one axis, exactly as lbm_halo_pack / _unpack do for the outer axis:
 *   axis: 0 = x, 1 = y, 2 = z (3-D only); side 0 / 1 = the low / high face of that axis,
 *         which must be a HALO face (LBM_ERR_ARG otherwise);
 *   buf: lbm_halo_axis_bytes(axis) bytes, packed as [direction][plane cell] fp32, momentum
 *        then thermal, directions with c_axis = +-1 in index order, plane cells with the
 *        lower remaining axis fastest (y then z for axis x; x then z for y; x then y for z).
 * The whole plane moves, the ghost rows of the other axes included.  Run the axes one after
 * another -- every pack and unpack of one axis before the next axis's packs, in the same
 * axis order at FILL and at DRAIN -- and a link across an edge or a corner reaches the
 * diagonal block in two or three hops through those rows: the FILL of the later axis
 * carries what the earlier one put in its ghost rows, and a DRAIN unpack writes a ghost row
 * of the other axis whenever the cell it lands in is one, from where the next axis's DRAIN
 * takes it on.  Between steps every owned cell then holds what one undivided domain would.
 * lbm_step_planes and the overlap above stay with the outer axis. */
lbm_status lbm_halo_axis_bytes(const lbm_ctx *ctx, int axis, size_t *bytes);
lbm_status lbm_halo_axis_pack(lbm_ctx *ctx, int axis, int side, int phase, void *buf);
lbm_status lbm_halo_axis_unpack(lbm_ctx *ctx, int axis, int side, int phase, const void *buf);

/* The exchange across one face of two blocks on the same device, without a buffer: lo's high
 * face of `axis` meets hi's low face.  One kernel moves both ways what lbm_halo_axis_pack on
 * one side and lbm_halo_axis_unpack on the other would move:
 *   FILL:  hi's first owned plane -> lo's ghost plane (directions with c_axis = +1), and lo's
 *          first owned plane -> hi's ghost plane (c_axis = -1);
 *   DRAIN: lo's ghost plane -> hi's first owned plane (c_axis = +1, wall links and solid cells
 *          of hi keep their slots), and hi's ghost plane -> lo's first owned plane (c_axis = -1).
 * lo and hi may be the same context (a ring of one block along that axis).  Both must be
 * initialised, at the same step, with the same lattices and equal extents on the other two
 * axes (LBM_ERR_ARG / LBM_ERR_STATE), and on one device (LBM_ERR_UNSUPPORTED otherwise).  The
 * kernel runs on lo's stream: work on hi issued on another stream must be ordered before the
 * call by the caller (an event), and later work on hi after it.  The parity rules are those of
 * the pack and unpack calls; the axis order rule for blocks holds as well. */
lbm_status lbm_halo_axis_swap(lbm_ctx *lo, lbm_ctx *hi, int axis, int phase);

/* n (1..32) face swaps of one axis in one launch: pair p swaps lo[p]'s high face with
 * hi[p]'s low face, as lbm_halo_axis_swap would, with its checks on every pair.  Every
 * context must be on one device, with the same lattices, at one step, and each face may
 * appear once (no context twice among lo[], nor twice among hi[]; LBM_ERR_ARG otherwise).
 * The swaps of one axis touch disjoint slots, so one launch equals the n calls in any
 * order.  Runs on lo[0]'s stream; work on the other contexts issued on other streams must
 * be ordered before the call by the caller.  lo and hi are host arrays of n pointers.
 * The error text of a failed call is lo[0]'s (lbm_last_error(lo[0])), or the thread's for
 * an n out of range. */
lbm_status lbm_halo_axis_swap_many(lbm_ctx *const *lo, lbm_ctx *const *hi, int n, int axis,
                                   int phase);

/* Enqueue later work on another stream (a cudaStream_t). */
lbm_status lbm_set_stream(lbm_ctx *ctx, void *cuda_stream);

/* Sum mass, momentum and thermal energy of populations held in caller memory, without
 * allocating anything.  No page describes this call: it is a service for callers that
 * cannot call cudaMalloc (code running inside another framework's memory pool, or in a
 * loop where an allocation is not allowed) and so cannot provide a workspace.
 *   f: Q planes (q-major) of nx*ny*nz fp32 populations, unshifted, in the lattice order
 *      above (as lbm_get_populations writes them); g: Q_T planes or NULL without thermal.
 *   out: 6 doubles written in stream order on cuda_stream (a cudaStream_t; NULL = legacy
 *      default stream): sum f, sum c_x f, sum c_y f, sum c_z f, sum g, and the number of
 *      cells whose sum f or sum g is not finite.  Nothing waits for the stream.
 *   f, g, out: device memory of the current device or page-locked host memory.
 * Limit: nx*ny*nz <= 2^28 (268435456) cells; larger grids are rejected with LBM_ERR_ARG,
 * as are D2Q9 grids with nz != 1.
 * The reduction's scratch is one file-scope static device array of 2 MiB, which every
 * device that loads the library keeps until the process exits.  The first call on a
 * device looks up that array's device address (once per device, with the device
 * current), so make a first call before capturing the stream into a CUDA graph.  Every
 * call reuses the same array: calls that overlap on the GPU (other streams, or threads
 * without ordering between them) race on it and must be serialised by the caller.
 * Errors are reported through lbm_last_error(NULL). */
lbm_status lbm_reduce_populations_static(int lattice, int thermal, int nx, int ny, int nz,
                                         const float *f, const float *g, double *out,
                                         void *cuda_stream);

int lbm_parity(const lbm_ctx *ctx);                 /* steps taken mod 2, -1 if ctx NULL */
long long lbm_steps_taken(const lbm_ctx *ctx);      /* -1 if ctx NULL                    */
const char *lbm_last_error(const lbm_ctx *ctx);     /* ctx NULL: last create-time error */
const char *lbm_version(void);
void lbm_destroy(lbm_ctx *ctx);                     /* frees the host context only       */

#ifdef __cplusplus
}
#endif
#endif
