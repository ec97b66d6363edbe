/*
 * hx.h - staged-forwarding halo exchange of a 3D domain decomposition, with
 * every domain held as a simulated rank in one GPU's memory (sm_103a).
 *
 * The operation is the GROMACS halo exchange described in "A Practical Guide
 * to GPU-Initiated Communication for Molecular Dynamics at Scale" (NVIDIA
 * technical blog):
 *   - coordinates: per pulse, the atoms listed by an index map are gathered
 *     from the sender's coordinate array and stored directly into the
 *     receiver's array at that pulse's receive offset; pulses run Z -> Y -> X
 *     and later pulses forward atoms received in earlier ones (intro; section
 *     "From MPI baseline to optimized GPU-native halo exchange"; section
 *     "Optimizing for efficient transfers across NVIDIA NVLink-connected
 *     GPUs" for the direct store into the peer's array);
 *   - forces: the same maps in reverse pulse order, accumulating received halo
 *     forces into the sender's force array (unpackRecvBufKernel<accumulate> in
 *     the MPI-baseline section; section "Force halo exchange: Reversing the
 *     dependency chain");
 *   - one fused launch per direction for all pulses, with per-pulse signals
 *     and a dependent tail that waits only for earlier pulses (sections
 *     "Enabling parallelism across pulses through kernel fusion" and
 *     "Dependency-aware packing"; signalPeerOnLastBlock for the last-block
 *     notification).
 *
 * Geometry (the pages leave it open; these readings fix it):
 *   orthorhombic periodic box L, n_d uniform slabs per dimension, domain id
 *   r = cx + nx*(cy + ny*cz); home cell c_d = min(n_d-1, floor(x_d*n_d/L_d))
 *   in fp64 on the fp32 input, home atoms in input order; only dimensions
 *   with n_d > 1 communicate, np_d = ceil(cutoff / (L_d/n_d)) pulses each,
 *   np_d < n_d required; in each pulse a domain sends to its lower neighbour
 *   (c_d - 1 mod n_d) the candidates x with (float)(x_d - lo_d) < (float)cutoff,
 *   lo_d = (float)(c_d*L_d/n_d) of the sender; candidates of pulse (d,0) are
 *   all local atoms, of pulse (d,k>0) the atoms received in (d,k-1); maps
 *   list local indices in ascending order; a sender in cell 0 adds (float)L_d
 *   to component d; forces are never shifted.
 *
 * Layout in the caller's flat float3 (AoS, 12 bytes per atom) buffers:
 *   domain r occupies slots [dom_offset[r], dom_offset[r] + home[r] + halo[r]):
 *   its home atoms, then the slots received in pulse 0, pulse 1, ... in the
 *   global pulse order. Coordinates and forces use the same layout.
 *
 * Conventions: every pointer argument is a device pointer unless marked
 * "host". `stream` is a cudaStream_t passed as void* (NULL = legacy default
 * stream). Calls are asynchronous on `stream` unless marked "synchronises".
 * A call that needs the handle's device makes it current for its duration
 * and gives the calling thread's current device back before it returns.
 * Return value: HX_OK (0) or a negative HX_ERR_* code; no call throws, and
 * there is no CPU fallback: a handle exists only on a working CUDA device.
 * The library owns the maps, tables, flags and graphs of a handle until
 * hx_destroy; the caller owns every buffer it passes in. A handle is not
 * thread-safe: calls on one handle must not run concurrently from several
 * host threads, and two exchanges of the same direction must not overlap on
 * the GPU (they share that direction's signal flags and epoch word). Successive
 * exchanges on one stream never do: under HX_FLAG_PDL the next kernel may be
 * scheduled early, but it waits for the previous one to complete before it
 * touches a flag or a buffer. Different handles are independent.
 */
#ifndef HX_H
#define HX_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct hx_ctx* hx_handle;

#define HX_OK 0
#define HX_ERR_ARG (-1)       /* null pointer, cutoff <= 0, dims < 1, box <= 0, bad index */
#define HX_ERR_PULSES (-2)    /* np_d >= n_d in some dimension, or too many pulses; from
                                 hx_build_maps also a plan beyond what the HX_FLAG_SWEEP_FORCES
                                 (8 pulses) or HX_FLAG_RESOLVED (7 copies per atom) tables hold */
#define HX_ERR_RANGE (-3)     /* an input position outside [0, L) or NaN */
#define HX_ERR_CAPACITY (-4)  /* caller buffer smaller than the layout needs */
#define HX_ERR_CUDA (-5)      /* a CUDA runtime call failed */
#define HX_ERR_TIMEOUT (-6)   /* a device-side wait for a pulse signal ran out of time */
#define HX_ERR_STATE (-7)     /* exchange before a successful hx_build_maps */
#define HX_ERR_NOMEM (-8)     /* host or device allocation failed */

/* hx_init flags */
#define HX_FLAG_UNORDERED_FORCES 0x1u /* force adds by atomics: order-free, within 1e-6 relative
                                          of the ordered result; default is ordered and bit-exact.
                                          Applies to the chunk force kernel: the slot sweep
                                          (HX_FLAG_SWEEP_FORCES) and resolved mode always add in
                                          order and ignore it */
#define HX_FLAG_NO_GRAPH 0x2u          /* launch the fused kernels directly, not through a CUDA graph */
#define HX_FLAG_FINE_WAITS 0x8u        /* chunk-granular dependencies: a chunk waits only for the
                                          chunks that wrote the slots it reads or, for forces, that
                                          add into its targets, each signalled by its own epoch flag;
                                          without it, the pages' per-pulse signals (the last chunk of
                                          a (sender, pulse) stores its epoch flag) */
#define HX_FLAG_SWEEP_FORCES 0x40u     /* the force exchange by the slot-sweep kernel: every warp
                                          takes units of up to 256 consecutive target slots of one
                                          sender, stages them, their map runs and their received
                                          force runs in shared memory with TMA bulk copies
                                          (cp.async.bulk), adds every pulse's contributions in
                                          reverse pulse order there and writes the slots back; per-
                                          unit signals; same results bit for bit. The coordinates
                                          stay on the chunk kernels. Not with HX_FLAG_RESOLVED (else
                                          HX_ERR_ARG); plans of more than 8 pulses get HX_ERR_PULSES
                                          from hx_build_maps */
#define HX_FLAG_BULK_STORE 0x200u      /* chunk coordinate kernels pack by bulk store: each warp gathers
                                          its chunk into shared memory and stores it to the receiver's
                                          slots with one cp.async.bulk (the pages' TMA variant, section
                                          "Optimizing for efficient transfers across NVIDIA
                                          NVLink-connected GPUs"); same results bit for bit. Applies
                                          where the chunk kernels run the coordinates */
#define HX_FLAG_PDL 0x400u             /* launch the exchange kernels directly with programmatic
                                          dependent launch, so an exchange may be scheduled while
                                          the stream's previous kernel finishes (it waits for that
                                          kernel before claiming work or touching coordinates,
                                          forces or flags; resolved kernels read their build-time
                                          tables first). A persistent grid lets the next kernel be
                                          scheduled only once all of its own blocks have started;
                                          with HX_FLAG_SWEEP_FORCES, only as the coordinate
                                          kernel's blocks exit, so that the sweep's grid lands on
                                          empty SMs and is wholly resident */
#define HX_FLAG_RESOLVED 0x100u        /* the forwarding unrolled at build time: every halo slot is
                                          gathered straight from its origin home atom (plus the
                                          shifts its path added), and every home atom's force tree
                                          (the atom and its copies) is summed in the staged order
                                          by one thread; one independent pass per direction, same
                                          results bit for bit. Forces are ordered
                                          (HX_FLAG_UNORDERED_FORCES is ignored); no device waits.
                                          A home atom may have at most 7 copies (else HX_ERR_PULSES
                                          from hx_build_maps), and a layout at most 2^29 slots (else
                                          HX_ERR_CAPACITY: a halo slot's origin and shifts share one
                                          32-bit word) */

#define HX_FLAGS_ALL 0x74bu      /* every flag above */

#define HX_MAX_PULSES 32
#define HX_MAX_DOMAINS 4096

/* Pulse plan of a decomposition without touching a GPU: validates the
 * arguments like hx_init and writes *n_pulses and, per global pulse p (Z
 * pulses first, then Y, then X), pulse_dim[p] (0=x,1=y,2=z) and pulse_k[p]
 * (index of the pulse within its dimension). pulse_dim/pulse_k are host
 * arrays of at least HX_MAX_PULSES entries and may be NULL.
 * Pages: "Dependency-aware packing" (global Z -> Y -> X numbering). */
int hx_query_plan(const double box[3], const int dims[3], double cutoff,
                  int* n_pulses, int32_t* pulse_dim, int32_t* pulse_k);

/* Creates a handle on CUDA device `device`. box (host, nm), dims (host),
 * cutoff (nm). timeout_us bounds every device-side wait for a pulse signal
 * (0 selects 1 s); a wait that runs out sets HX_ERR_TIMEOUT, read by
 * hx_status, and the kernel still finishes. flags: HX_FLAG_* above; a bit
 * outside them is HX_ERR_ARG. Errors: HX_ERR_ARG, HX_ERR_PULSES, HX_ERR_CUDA
 * (no usable device), HX_ERR_NOMEM.
 * Pages: the pulse plan of "Dependency-aware packing" (Z -> Y -> X, one
 * pulse per dimension when the cutoff fits one neighbour, more otherwise);
 * the box, slab and cutoff geometry is not on the pages (readings above). */
int hx_init(hx_handle* out, const double box[3], const int dims[3], double cutoff,
            int device, unsigned flags, unsigned timeout_us);

/* Builds the decomposition on the GPU from pos_in (device, fp32 [n_atoms][3],
 * any order): home cells, stable home partition, then pulse by pulse in the
 * global order the cutoff selection with stable compaction into ascending
 * maps, the receive offsets and the forwarded coordinates (the maps are the
 * inputs of every kernel on the pages: packSendBufKernel's `map`, the fused
 * kernel's `indexMap`). Writes *needed (host) = slots of the layout. If
 * coords (device, float3 slots) is non-NULL and capacity >= *needed, it also
 * writes every domain's home coordinates and fills every halo slot (one
 * coordinate exchange). coords == NULL only sizes the layout (maps are kept);
 * capacity < *needed returns HX_ERR_CAPACITY with the maps kept and coords
 * untouched. Synchronises `stream` once per pulse to read sizes. Resets all
 * pulse signals. Errors: HX_ERR_ARG, HX_ERR_RANGE, HX_ERR_CAPACITY,
 * HX_ERR_CUDA, HX_ERR_NOMEM. */
int hx_build_maps(hx_handle h, const float* pos_in, int64_t n_atoms,
                  float* coords, int64_t capacity, int64_t* needed, void* stream);

/* Sizes after a build (host outputs; any may be NULL): domains, pulses,
 * slots of the layout, map entries. Not on the pages (they take the maps'
 * sizes as given: packSendBufKernel's `size`, the fused kernel's per-pulse
 * send sizes); this reports what hx_build_maps derived. */
int hx_get_counts(hx_handle h, int* n_domains, int* n_pulses, int64_t* total_slots,
                  int64_t* total_entries);

/* Resolved mode's force trees after a build (host outputs; any may be
 * NULL): trees that are an atom and one copy (one add), corner trees of four
 * nodes summed in a fixed order (three adds), and general trees. All three
 * are 0 for a handle without HX_FLAG_RESOLVED. Errors: HX_ERR_ARG,
 * HX_ERR_STATE. */
int hx_get_resolved_counts(hx_handle h, int64_t* n_pairs, int64_t* n_quads, int64_t* n_general);

/* Per-domain layout (host arrays of n_domains entries; any may be NULL):
 * first slot, home-atom count, halo-slot count. Pages: "From MPI baseline to
 * optimized GPU-native halo exchange" (received halo data lands in the
 * coordinate buffer at its offset after the home atoms; the fused kernel's
 * atomOffsetInPeer). */
int hx_get_layout(hx_handle h, int64_t* dom_offset, int32_t* home_count, int32_t* halo_count);

/* home_ids (device, int32 [n_atoms]): for the k-th home slot in layout order
 * (domain 0's home atoms, then domain 1's, ...) the input index of its atom.
 * Not on the pages (their ranks own their atoms from the start); it maps the
 * layout back to the caller's input order. */
int hx_get_home_ids(hx_handle h, int32_t* home_ids, void* stream);

/* Copies the maps to host for inspection (synchronises). maps_host (host,
 * int32, cap entries >= total_entries) receives every map, pulse-major then
 * sender-minor; table_host (host, int64 [n_pulses][n_domains][6]) receives
 * per (pulse, sender): map offset, size, receiving domain, receive offset in
 * the receiver's array, shift flag (1 when the sender adds L_d), and the
 * length of the independent prefix (entries whose local index is below the
 * sender's home count, the pages' dependencyAtomOffset split). Either may be
 * NULL. HX_ERR_CAPACITY if cap < total_entries. */
int hx_get_maps(hx_handle h, int32_t* maps_host, int64_t cap, int64_t* table_host);

/* Coordinate exchange, in place on coords (device, float3 slots of the
 * layout): for every pulse Z -> Y -> X, coords[receiver slot i] =
 * coords[sender slot map[i]] (+L_d when shifted). One persistent kernel for
 * all pulses: independent entries are stored at once, the forwarded tail of
 * a pulse waits (acquire, gpu scope) for the signals of earlier pulses, and
 * each (sender, pulse) is signalled (release, gpu scope) when all its chunks
 * are stored. Pages: packSendBufKernel, packHaloCoords, packSubset,
 * fusedPulsesPackAndSendKernel, signalPeerOnLastBlock. */
int hx_exchange_coords(hx_handle h, float* coords, void* stream);

/* Force exchange, in place on forces (device, float3 slots of the layout):
 * for every pulse X -> Y -> Z (reverse), forces[sender slot map[i]] +=
 * forces[receiver slot i], fp32, x then y then z. One persistent kernel; a
 * (sender, pulse) starts once every later pulse that touches its targets or
 * its source slots has signalled, so each home force is the fp32 sum in
 * reverse pulse order (bit-exact) unless HX_FLAG_UNORDERED_FORCES. Halo slots
 * keep their values except where they forward accumulated forces. Pages:
 * unpackRecvBufKernel<accumulate=true>; "Force halo exchange: Reversing the
 * dependency chain". */
int hx_exchange_forces(hx_handle h, float* forces, void* stream);

/* The two exchanges for data that lives in host memory: each copies the
 * direction's inputs in, runs the exchange above on the device buffer, and
 * copies its results out, all queued on `stream` (the host buffer holds the
 * results once the stream has passed this point). The pages keep all data on
 * the GPU ("From MPI baseline to optimized GPU-native halo exchange" names
 * the CPU hand-offs as the cost); these calls only add the host copies.
 *   host: float3 slots of the layout in page-locked host memory that is
 *         mapped for the device (cudaHostAlloc, or cudaHostRegister with
 *         cudaHostRegisterMapped); total_slots slots, owned by the caller.
 *   dev:  device float3 slots of the layout, owned by the caller; its halo
 *         (coordinates) or all (forces) slots are overwritten.
 * hx_exchange_coords_host: every domain's home coordinates host -> dev,
 *   hx_exchange_coords(dev), every domain's halo slots dev -> host.
 *   Host traffic: 12 B per home slot in, 12 B per halo slot out.
 * hx_exchange_forces_host: every slot's force host -> dev,
 *   hx_exchange_forces(dev), every domain's home forces dev -> host.
 *   Host traffic: 12 B per slot in, 12 B per home slot out.
 * The copies run on the SMs through the mapped host buffer (one launch per
 * direction for all domains' ranges), except the forces' single
 * contiguous copy in. Errors: those of the exchange, and HX_ERR_ARG for a
 * NULL buffer or a host buffer that is not mapped page-locked memory. */
int hx_exchange_coords_host(hx_handle h, float* coords_host, float* coords_dev, void* stream);
int hx_exchange_forces_host(hx_handle h, float* forces_host, float* forces_dev, void* stream);

/* The same two exchanges with packed host buffers: a domain's atoms are
 * contiguous in host memory, so each direction crosses the host link as one
 * copy-engine transfer, and the scatter into the slot layout and the gather
 * out of it run as range copies in HBM (like the pages' packSendBufKernel,
 * which gathers a pulse's atoms into one contiguous buffer before it is sent;
 * "From MPI baseline to optimized GPU-native halo exchange").
 *   hx_exchange_coords_host_packed: home_host (host, float3 [n_atoms]) holds
 *     the home coordinates in layout order (domain 0's home slots, then
 *     domain 1's, ...: the order of hx_get_home_ids); they are copied into
 *     coords_dev's home slots, hx_exchange_coords(coords_dev) runs, and every
 *     halo slot is copied out to halo_host (host, float3 [total_slots -
 *     n_atoms]) in layout order (domain 0's halo slots, then domain 1's, ...).
 *   hx_exchange_forces_host_packed: forces_host (host, float3 slots of the
 *     layout: every slot's force) is copied into forces_dev,
 *     hx_exchange_forces(forces_dev) runs, and the home forces are copied out
 *     to home_forces_host (host, float3 [n_atoms], layout order).
 *   coords_dev / forces_dev: device float3 slots of the layout, owned by the
 *     caller (as for the calls above).
 * All copies are queued on `stream`; the output buffer holds the results once
 * the stream has passed this point. Host buffers should be page-locked
 * (cudaHostAlloc or cudaHostRegister) for the copies to be asynchronous;
 * pageable memory gives the same results with synchronous copies. They are
 * owned by the caller and must not be written (input) or read (output) until
 * the stream has passed the call. Host traffic: 12 B per home slot in and
 * 12 B per halo slot out (coordinates), 12 B per slot in and 12 B per home
 * slot out (forces), as for the calls above. The first packed call after a
 * build allocates the handle's packing buffer (12 B x the larger of the home
 * and halo slot counts), kept until the next build or hx_destroy; make it
 * before any stream capture. Calls on one handle share that buffer: calls
 * whose work overlaps on the GPU (other streams) race, so use one handle per
 * stream. Errors: those of the exchange; HX_ERR_ARG for a NULL buffer that
 * would be read or written; HX_ERR_NOMEM if the buffer cannot be allocated. */
int hx_exchange_coords_host_packed(hx_handle h, const float* home_host, float* halo_host, float* coords_dev,
                                   void* stream);
int hx_exchange_forces_host_packed(hx_handle h, const float* forces_host, float* home_forces_host,
                                   float* forces_dev, void* stream);

/* Unfused baseline of the same two exchanges: one stream-ordered kernel
 * launch per pulse (all senders of that pulse in one launch), no signals.
 * Same results bit for bit as the fused calls in ordered mode. Pages: the
 * per-pulse packSendBufKernel / unpackRecvBufKernel loop of the MPI
 * baseline, with the host synchronisations replaced by stream order. */
int hx_exchange_coords_unfused(hx_handle h, float* coords, void* stream);
int hx_exchange_forces_unfused(hx_handle h, float* forces, void* stream);

/* Same as hx_exchange_coords, for callers that must not allocate device
 * memory while they run (an engine that reserves all GPU memory for its own
 * arena, or code that may only use memory it has accounted for). The pages
 * have no counterpart: this concerns how the library holds its scratch.
 * The call never allocates: the kernel's signal flags, election counters and
 * control block live in one fixed file-scope device array of
 * HX_STATIC_MAX_FLAGS flags (about 1.5 MB, held by every GPU that loads the
 * library until the process exits), cleared on `stream` at each call, and
 * the kernel is launched directly, without a CUDA graph. hx_build_maps does
 * the set-up, with the handle's device current: it looks up that array's
 * device address (cudaGetSymbolAddress) and loads the kernel this call
 * launches, so the call itself only reads the handle. All calls share the
 * one array, which keeps the last call's contents, so calls whose work
 * overlaps on the GPU (other streams, other handles on the same device)
 * race: serialise them. A device-side time-out of this call is reported by
 * hx_status of the calling handle (after the stream this call ran on has
 * passed it) until another handle makes a static call on the same device or
 * hx_clear_status clears it. Errors: HX_ERR_ARG, HX_ERR_STATE, HX_ERR_CUDA
 * (also when the build could not do the set-up), and HX_ERR_CAPACITY when
 * the handle's work list needs more than HX_STATIC_MAX_FLAGS signal flags
 * (its item count or chunk count, whichever it signals by); nothing is
 * launched then. */
#define HX_STATIC_MAX_FLAGS 131072
int hx_exchange_coords_static(hx_handle h, float* coords, void* stream);

/* Launches one empty kernel the way the fused exchanges are launched (graph,
 * direct, or direct with programmatic dependent launch, per the handle's
 * flags): the launch floor for latency measurements. Not on the pages; it measures the per-launch cost that
 * "Strategies in a nutshell" (six launches fused into one) removes. */
int hx_noop(hx_handle h, void* stream);

/* Synchronises `stream` and returns the sticky device status: HX_OK or
 * HX_ERR_TIMEOUT (a wait for a pulse signal ran out). *detail (host, may be
 * NULL) receives direction*65536 + item (item = pulse*n_domains + sender)
 * of the first wait that gave up, or -1. The regular exchanges' status comes
 * first; then that of the handle's last hx_exchange_coords_static call, if
 * no other handle has made one on the device since. Not on the pages (their
 * signal waits are unbounded); the bounded wait and its status are the
 * failure detection of this library. */
int hx_status(hx_handle h, void* stream, int* detail);

/* The regular exchanges' sticky status without synchronising: queues on
 * `stream` one small kernel that reads it and a copy of {status, detail}
 * (as hx_status returns them; HX_OK and -1 when no wait gave up) into
 * status_host[0] and status_host[1] (host memory owned by the caller;
 * page-locked for the copy to be asynchronous). The values are there once
 * the stream has passed this point, e.g. after an event recorded after the
 * call, so a caller can check every step for a time-out without stalling the
 * stream. A call between two exchanges on the stream sits between their
 * launches (no programmatic overlap there). The static path's status is read
 * by hx_status only. Not on the pages (their waits are unbounded). Errors:
 * HX_ERR_ARG (NULL handle or buffer), HX_ERR_CUDA. */
int hx_status_async(hx_handle h, int* status_host, void* stream);

/* Synchronises `stream`, clears the status (the handle's, and the static
 * path's when hx_status would report it) and resets every pulse signal,
 * counter and epoch so that the next exchange starts clean. Not on the
 * pages: the recovery half of hx_status. */
int hx_clear_status(hx_handle h, void* stream);

/* Fault injection for tests (host side, no device fault): the chunks of
 * (direction 0 = coordinates / 1 = forces, domain, pulse) stop signalling,
 * so its waiters run into the timeout. domain = -1 switches it off. */
int hx_debug_drop_signal(hx_handle h, int direction, int domain, int pulse);

/* Test and tuning hook for the force sweep (HX_FLAG_SWEEP_FORCES): mode 1
 * makes each dependent segment of a unit wait for its own producers (the
 * default where a warp has at most four units), mode 2 makes a unit wait for
 * all its producers before staging (the default otherwise), mode 0 restores
 * the automatic choice. Results are bit-identical in every mode; only the
 * timing differs. Synchronises the device and drops the handle's cached
 * graphs. Not on the pages (their force kernel waits per pulse). Errors:
 * HX_ERR_ARG, HX_ERR_CUDA. */
int hx_debug_sweep_waits(hx_handle h, int mode);

/* Human-readable name of an HX_* code (static string). Not on the pages. */
const char* hx_error_string(int code);

/* Frees everything the handle owns (synchronises its device). NULL is a no-op.
 * Not on the pages (resource lifetime of this library). */
void hx_destroy(hx_handle h);

#ifdef __cplusplus
}
#endif

#endif /* HX_H */
