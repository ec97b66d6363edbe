/*
 * CPU oracle for the staged-forwarding halo exchange of a 3D domain
 * decomposition.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path links, loads or calls
 * this file: only the tests, the smoke check in __graft_entry__ and the CPU
 * baseline leg of bench.py use it. It shares no code, header, table or
 * constant generator with the CUDA library.
 *
 * What it computes follows "A Practical Guide to GPU-Initiated Communication
 * for Molecular Dynamics at Scale" (NVIDIA technical blog):
 *   - staged forwarding: boundary atoms are relayed through intermediate
 *     domains, dimension by dimension, in one or more pulses; coordinates go
 *     Z, then Y, then X (intro, and section "From MPI baseline to optimized
 *     GPU-native halo exchange");
 *   - a pulse packs the atoms listed by an index map into the receiver's
 *     coordinate array at that pulse's receive offset: packed[i] =
 *     data[map[i]] (packSendBufKernel in the same section; the received data
 *     "lands directly in the coordinate buffer at the correct offset");
 *   - forces travel back in the reverse order and are accumulated through
 *     the same map: forces[map[i]] += packed[i] (unpackRecvBufKernel, and
 *     section "Force halo exchange: Reversing the dependency chain");
 *   - pulses are numbered globally Z -> Y -> X and a pulse's forwarded
 *     (dependent) atoms are those whose local index is at or above the
 *     sender's home-atom count (section "Enabling parallelism across pulses
 *     through kernel fusion", the dependencyAtomOffset split).
 *
 * The pages leave the geometry open; this oracle takes these readings:
 *   - orthorhombic periodic box L, uniform slabs n_d per dimension, domain id
 *     r = cx + nx*(cy + ny*cz);
 *   - home cell c_d = min(n_d-1, floor(x_d * n_d / L_d)) evaluated in fp64 on
 *     the fp32 input; home atoms keep input order;
 *   - lower slab face lo_d(c) = (float)(c * L_d / n_d) in fp64 then rounded;
 *   - only dimensions with n_d > 1 communicate, with np_d = ceil(r_c / w_d)
 *     pulses (w_d = L_d / n_d); np_d < n_d is required;
 *   - in every pulse of dimension d a domain sends to its lower neighbour
 *     (c_d - 1 mod n_d) and receives from its upper neighbour;
 *   - candidates of pulse (d, 0) are all local atoms of the sender (home plus
 *     everything received in earlier dimensions); candidates of pulse (d, k>0)
 *     are only the atoms received in pulse (d, k-1);
 *   - an atom is sent when (float)(x_d - lo_d(c_sender)) < (float)r_c, one
 *     fp32 subtraction, strict comparison, in the sender's frame;
 *   - the map lists selected local indices in ascending order;
 *   - a sender in cell c_d == 0 adds (float)L_d to component d of every
 *     packed coordinate (periodic shift); forces are never shifted;
 *   - a domain's array is [home | recv pulse 0 | recv pulse 1 | ...];
 *   - the force exchange visits pulses last to first and adds in fp32,
 *     component by component.
 *
 * Compile with -ffp-contract=off (there is no multiply in the exchanged
 * arithmetic, but the flag keeps the reading "one IEEE fp32 add or subtract
 * per operation" independent of the compiler). With -fopenmp the *_par
 * exchanges run each pulse's senders on several threads, pulse order kept:
 * the same arithmetic on independent senders, used to time the oracle on all
 * host cores.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OR_OK 0
#define OR_ERR_ARG (-1)
#define OR_ERR_PULSES (-2)
#define OR_ERR_RANGE (-3)
#define OR_ERR_MEM (-8)
#define OR_MAX_PULSES 64

typedef struct {
    float* v;      /* xyz triples */
    int64_t len;   /* atoms */
    int64_t cap;
} farr;

typedef struct {
    double box[3];
    int dims[3];
    double cutoff;
    float boxf[3];
    float rcf;
    int np[3];
    int n_pulses;
    int pulse_dim[OR_MAX_PULSES];
    int pulse_k[OR_MAX_PULSES];
    float* lo[3];
    int ndom;

    int built;
    int64_t n_atoms;
    int32_t* home;        /* [ndom] home-atom count */
    int32_t* halo;        /* [ndom] halo-slot count */
    int64_t* dom_offset;  /* [ndom] first slot of each domain in the flat array */
    int32_t* home_ids;    /* [n_atoms] input index of each home slot, layout order */
    int64_t total_slots;
    /* per (pulse p, sender r), index p*ndom + r */
    int64_t* t_map_off;
    int32_t* t_size;
    int32_t* t_recv;      /* receiving domain */
    int32_t* t_off;       /* receive offset inside the receiver's array */
    int32_t* t_shift;     /* 1 when the sender adds L_d */
    int32_t* t_split;     /* entries with local index < home count (a prefix) */
    int32_t* maps;
    int64_t total_entries;
    float* coords;        /* [total_slots*3] array produced by the build */
} oracle_dd;

static void cell_of_domain(const oracle_dd* o, int r, int c[3]) {
    c[0] = r % o->dims[0];
    c[1] = (r / o->dims[0]) % o->dims[1];
    c[2] = r / (o->dims[0] * o->dims[1]);
}

static int domain_of_cell(const oracle_dd* o, const int c[3]) {
    return c[0] + o->dims[0] * (c[1] + o->dims[1] * c[2]);
}

/* Lower neighbour along d: the domain that receives from r in a pulse of d. */
static int lower_neighbour(const oracle_dd* o, int r, int d) {
    int c[3];
    cell_of_domain(o, r, c);
    c[d] = (c[d] - 1 + o->dims[d]) % o->dims[d];
    return domain_of_cell(o, c);
}

static void free_build(oracle_dd* o) {
    free(o->home); free(o->halo); free(o->dom_offset); free(o->home_ids);
    free(o->t_map_off); free(o->t_size); free(o->t_recv); free(o->t_off);
    free(o->t_shift); free(o->t_split); free(o->maps); free(o->coords);
    o->home = o->halo = NULL; o->dom_offset = NULL; o->home_ids = NULL;
    o->t_map_off = NULL; o->t_size = o->t_recv = o->t_off = o->t_shift = o->t_split = NULL;
    o->maps = NULL; o->coords = NULL;
    o->built = 0;
}

void oracle_destroy(oracle_dd* o) {
    if (!o) return;
    free_build(o);
    for (int d = 0; d < 3; ++d) free(o->lo[d]);
    free(o);
}

/* Set-up: widths, pulse counts, the global pulse order Z, Y, X and the fp32
 * lower-face table. Returns NULL and *err on invalid input. */
oracle_dd* oracle_create(const double box[3], const int dims[3], double cutoff, int* err) {
    *err = OR_OK;
    if (!box || !dims || !(cutoff > 0.0) || !isfinite(cutoff)) { *err = OR_ERR_ARG; return NULL; }
    for (int d = 0; d < 3; ++d) {
        if (dims[d] < 1 || !(box[d] > 0.0) || !isfinite(box[d])) { *err = OR_ERR_ARG; return NULL; }
    }
    oracle_dd* o = (oracle_dd*)calloc(1, sizeof(oracle_dd));
    if (!o) { *err = OR_ERR_MEM; return NULL; }
    o->cutoff = cutoff;
    o->rcf = (float)cutoff;
    o->ndom = 1;
    for (int d = 0; d < 3; ++d) {
        o->box[d] = box[d];
        o->dims[d] = dims[d];
        o->boxf[d] = (float)box[d];
        o->ndom *= dims[d];
        if (dims[d] > 1) {
            double w = box[d] / dims[d];
            o->np[d] = (int)ceil(cutoff / w);
            if (o->np[d] >= dims[d]) { *err = OR_ERR_PULSES; oracle_destroy(o); return NULL; }
        } else {
            o->np[d] = 0;
        }
        o->lo[d] = (float*)malloc(sizeof(float) * (size_t)dims[d]);
        if (!o->lo[d]) { *err = OR_ERR_MEM; oracle_destroy(o); return NULL; }
        for (int c = 0; c < dims[d]; ++c) o->lo[d][c] = (float)((double)c * box[d] / dims[d]);
    }
    int p = 0;
    for (int d = 2; d >= 0; --d) {          /* Z first, then Y, then X */
        for (int k = 0; k < o->np[d]; ++k) {
            if (p >= OR_MAX_PULSES) { *err = OR_ERR_PULSES; oracle_destroy(o); return NULL; }
            o->pulse_dim[p] = d;
            o->pulse_k[p] = k;
            ++p;
        }
    }
    o->n_pulses = p;
    return o;
}

int oracle_num_pulses(const oracle_dd* o) { return o->n_pulses; }
int oracle_num_domains(const oracle_dd* o) { return o->ndom; }
void oracle_pulse_list(const oracle_dd* o, int32_t* dim, int32_t* k) {
    for (int p = 0; p < o->n_pulses; ++p) { dim[p] = o->pulse_dim[p]; k[p] = o->pulse_k[p]; }
}
void oracle_lo_table(const oracle_dd* o, int d, float* out) {
    for (int c = 0; c < o->dims[d]; ++c) out[c] = o->lo[d][c];
}

static int farr_push(farr* a, const float v[3]) {
    if (a->len == a->cap) {
        int64_t nc = a->cap ? 2 * a->cap : 64;
        float* nv = (float*)realloc(a->v, sizeof(float) * 3 * (size_t)nc);
        if (!nv) return OR_ERR_MEM;
        a->v = nv;
        a->cap = nc;
    }
    a->v[3 * a->len + 0] = v[0];
    a->v[3 * a->len + 1] = v[1];
    a->v[3 * a->len + 2] = v[2];
    a->len += 1;
    return OR_OK;
}

/* Home layout, maps and the filled coordinate array, pulse by pulse in the
 * global order. */
int oracle_build(oracle_dd* o, const float* pos, int64_t n) {
    free_build(o);
    const int ndom = o->ndom;
    const int P = o->n_pulses;
    int rc = OR_OK;
    if (n < 0 || (n > 0 && !pos)) return OR_ERR_ARG;

    /* 1. home cell of every atom (fp64 floor on the fp32 input) */
    int32_t* dom = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n > 0 ? n : 1));
    o->home = (int32_t*)calloc((size_t)ndom, sizeof(int32_t));
    o->halo = (int32_t*)calloc((size_t)ndom, sizeof(int32_t));
    o->dom_offset = (int64_t*)calloc((size_t)ndom, sizeof(int64_t));
    o->home_ids = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n > 0 ? n : 1));
    farr* local = (farr*)calloc((size_t)ndom, sizeof(farr));
    int64_t* off = (int64_t*)calloc((size_t)ndom * (size_t)(P > 0 ? P : 1), sizeof(int64_t));
    int64_t* rcv = (int64_t*)calloc((size_t)ndom * (size_t)(P > 0 ? P : 1), sizeof(int64_t));
    int32_t** pmap = (int32_t**)calloc((size_t)ndom * (size_t)(P > 0 ? P : 1), sizeof(int32_t*));
    int64_t* psize = (int64_t*)calloc((size_t)ndom * (size_t)(P > 0 ? P : 1), sizeof(int64_t));
    int64_t* snap = (int64_t*)calloc((size_t)ndom, sizeof(int64_t));
    if (!dom || !o->home || !o->halo || !o->dom_offset || !o->home_ids || !local || !off || !rcv ||
        !pmap || !psize || !snap) { rc = OR_ERR_MEM; goto done; }

    for (int64_t i = 0; i < n; ++i) {
        int c[3];
        for (int d = 0; d < 3; ++d) {
            double x = (double)pos[3 * i + d];
            if (!(x >= 0.0 && x < o->box[d])) { rc = OR_ERR_RANGE; goto done; }
            int cd = (int)floor(x * (double)o->dims[d] / o->box[d]);
            if (cd > o->dims[d] - 1) cd = o->dims[d] - 1;
            c[d] = cd;
        }
        dom[i] = domain_of_cell(o, c);
    }

    /* 2. stable partition: home atoms of each domain in input order */
    for (int64_t i = 0; i < n; ++i) o->home[dom[i]] += 1;
    {
        int64_t* fill = (int64_t*)calloc((size_t)ndom, sizeof(int64_t));
        if (!fill) { rc = OR_ERR_MEM; goto done; }
        int64_t s = 0;
        for (int r = 0; r < ndom; ++r) { fill[r] = s; s += o->home[r]; }
        for (int64_t i = 0; i < n; ++i) {
            int r = dom[i];
            o->home_ids[fill[r]++] = (int32_t)i;
            if ((rc = farr_push(&local[r], &pos[3 * i])) != OR_OK) { free(fill); goto done; }
        }
        free(fill);
    }

    /* 3. pulses in global order */
    for (int p = 0; p < P; ++p) {
        const int d = o->pulse_dim[p];
        const int k = o->pulse_k[p];
        for (int r = 0; r < ndom; ++r) snap[r] = local[r].len;
        for (int r = 0; r < ndom; ++r) {
            int c[3];
            cell_of_domain(o, r, c);
            const float lo = o->lo[d][c[d]];
            int64_t cb, ce;
            if (k == 0) { cb = 0; ce = snap[r]; }
            else { cb = off[(size_t)r * P + (p - 1)]; ce = cb + rcv[(size_t)r * P + (p - 1)]; }
            int64_t cnt = 0;
            int32_t* m = (int32_t*)malloc(sizeof(int32_t) * (size_t)(ce - cb > 0 ? ce - cb : 1));
            if (!m) { rc = OR_ERR_MEM; goto done; }
            for (int64_t j = cb; j < ce; ++j) {
                float rel = local[r].v[3 * j + d] - lo;
                if (rel < o->rcf) m[cnt++] = (int32_t)j;
            }
            pmap[(size_t)r * P + p] = m;
            psize[(size_t)r * P + p] = cnt;
        }
        for (int r = 0; r < ndom; ++r) {
            int c[3];
            cell_of_domain(o, r, c);
            const int q = lower_neighbour(o, r, d);
            const int shift = (c[d] == 0);
            const int32_t* m = pmap[(size_t)r * P + p];
            const int64_t S = psize[(size_t)r * P + p];
            off[(size_t)q * P + p] = snap[q];
            rcv[(size_t)q * P + p] = S;
            for (int64_t i = 0; i < S; ++i) {
                float v[3];
                v[0] = local[r].v[3 * (int64_t)m[i] + 0];
                v[1] = local[r].v[3 * (int64_t)m[i] + 1];
                v[2] = local[r].v[3 * (int64_t)m[i] + 2];
                if (shift) v[d] = v[d] + o->boxf[d];
                if ((rc = farr_push(&local[q], v)) != OR_OK) goto done;
            }
        }
    }

    /* 4. flat layout, table and maps (pulse-major, sender-minor) */
    {
        int64_t s = 0;
        for (int r = 0; r < ndom; ++r) {
            o->dom_offset[r] = s;
            o->halo[r] = (int32_t)(local[r].len - o->home[r]);
            s += local[r].len;
        }
        o->total_slots = s;
        int64_t e = 0;
        for (int p = 0; p < P; ++p)
            for (int r = 0; r < ndom; ++r) e += psize[(size_t)r * P + p];
        o->total_entries = e;
        size_t nt = (size_t)ndom * (size_t)(P > 0 ? P : 1);
        o->t_map_off = (int64_t*)calloc(nt, sizeof(int64_t));
        o->t_size = (int32_t*)calloc(nt, sizeof(int32_t));
        o->t_recv = (int32_t*)calloc(nt, sizeof(int32_t));
        o->t_off = (int32_t*)calloc(nt, sizeof(int32_t));
        o->t_shift = (int32_t*)calloc(nt, sizeof(int32_t));
        o->t_split = (int32_t*)calloc(nt, sizeof(int32_t));
        o->maps = (int32_t*)malloc(sizeof(int32_t) * (size_t)(e > 0 ? e : 1));
        o->coords = (float*)malloc(sizeof(float) * 3 * (size_t)(s > 0 ? s : 1));
        if (!o->t_map_off || !o->t_size || !o->t_recv || !o->t_off || !o->t_shift || !o->t_split ||
            !o->maps || !o->coords) { rc = OR_ERR_MEM; goto done; }
        int64_t mo = 0;
        for (int p = 0; p < P; ++p) {
            const int d = o->pulse_dim[p];
            for (int r = 0; r < ndom; ++r) {
                int c[3];
                cell_of_domain(o, r, c);
                const size_t t = (size_t)p * ndom + r;
                const int q = lower_neighbour(o, r, d);
                const int64_t S = psize[(size_t)r * P + p];
                const int32_t* m = pmap[(size_t)r * P + p];
                o->t_map_off[t] = mo;
                o->t_size[t] = (int32_t)S;
                o->t_recv[t] = q;
                o->t_off[t] = (int32_t)off[(size_t)q * P + p];
                o->t_shift[t] = (c[d] == 0);
                int32_t split = 0;
                for (int64_t i = 0; i < S; ++i) {
                    o->maps[mo + i] = m[i];
                    if (m[i] < o->home[r]) split = (int32_t)(i + 1);
                }
                o->t_split[t] = split;
                mo += S;
            }
        }
        for (int r = 0; r < ndom; ++r)
            memcpy(o->coords + 3 * o->dom_offset[r], local[r].v, sizeof(float) * 3 * (size_t)local[r].len);
    }
    o->n_atoms = n;
    o->built = 1;

done:
    if (local) for (int r = 0; r < ndom; ++r) free(local[r].v);
    if (pmap) for (size_t t = 0; t < (size_t)ndom * (size_t)(P > 0 ? P : 1); ++t) free(pmap[t]);
    free(local); free(pmap); free(psize); free(off); free(rcv); free(snap); free(dom);
    if (rc != OR_OK) free_build(o);
    return rc;
}

int64_t oracle_total_slots(const oracle_dd* o) { return o->built ? o->total_slots : -1; }
int64_t oracle_total_entries(const oracle_dd* o) { return o->built ? o->total_entries : -1; }

void oracle_get_layout(const oracle_dd* o, int64_t* dom_offset, int32_t* home, int32_t* halo) {
    for (int r = 0; r < o->ndom; ++r) {
        dom_offset[r] = o->dom_offset[r];
        home[r] = o->home[r];
        halo[r] = o->halo[r];
    }
}

void oracle_get_home_ids(const oracle_dd* o, int32_t* ids) {
    memcpy(ids, o->home_ids, sizeof(int32_t) * (size_t)o->n_atoms);
}

/* table row per (p, r): map_off, size, receiver, recv offset, shift, split */
void oracle_get_maps(const oracle_dd* o, int32_t* maps, int64_t* table) {
    memcpy(maps, o->maps, sizeof(int32_t) * (size_t)o->total_entries);
    for (size_t t = 0; t < (size_t)o->n_pulses * (size_t)o->ndom; ++t) {
        table[6 * t + 0] = o->t_map_off[t];
        table[6 * t + 1] = o->t_size[t];
        table[6 * t + 2] = o->t_recv[t];
        table[6 * t + 3] = o->t_off[t];
        table[6 * t + 4] = o->t_shift[t];
        table[6 * t + 5] = o->t_split[t];
    }
}

void oracle_get_coords(const oracle_dd* o, float* coords) {
    memcpy(coords, o->coords, sizeof(float) * 3 * (size_t)o->total_slots);
}

/* Coordinate exchange on a flat array whose home slots hold current
 * coordinates: replay every pulse in order; packed[i] = data[map[i]], with
 * the periodic shift, stored at the receiver's offset.
 *
 * `threads` > 1 runs the senders of one pulse on that many OpenMP threads
 * (pulse order kept). Within a pulse every sender writes only its own
 * receiver's receive range of that pulse, and reads only its home and
 * earlier receive ranges, so no two senders touch the same slot and the
 * result is the same bit for bit. */
static void exchange_coords_impl(const oracle_dd* o, float* x, int threads) {
    (void)threads;
    for (int p = 0; p < o->n_pulses; ++p) {
        const int d = o->pulse_dim[p];
#ifdef _OPENMP
#pragma omp parallel for num_threads(threads) schedule(dynamic, 1) if (threads > 1)
#endif
        for (int r = 0; r < o->ndom; ++r) {
            const size_t t = (size_t)p * o->ndom + r;
            const int32_t* m = o->maps + o->t_map_off[t];
            const int64_t S = o->t_size[t];
            const float* src = x + 3 * o->dom_offset[r];
            float* dst = x + 3 * (o->dom_offset[o->t_recv[t]] + o->t_off[t]);
            for (int64_t i = 0; i < S; ++i) {
                float v0 = src[3 * (int64_t)m[i] + 0];
                float v1 = src[3 * (int64_t)m[i] + 1];
                float v2 = src[3 * (int64_t)m[i] + 2];
                if (o->t_shift[t]) {
                    if (d == 0) v0 = v0 + o->boxf[0];
                    else if (d == 1) v1 = v1 + o->boxf[1];
                    else v2 = v2 + o->boxf[2];
                }
                dst[3 * i + 0] = v0;
                dst[3 * i + 1] = v1;
                dst[3 * i + 2] = v2;
            }
        }
    }
}

/* Force exchange: pulses last to first; forces[map[i]] += received[i].
 * With `threads` > 1 the senders of one pulse run in parallel: a sender adds
 * only into its own home and earlier receive ranges and reads its receiver's
 * receive range of this pulse, which no sender writes in this pulse. */
static void exchange_forces_impl(const oracle_dd* o, float* f, int threads) {
    (void)threads;
    for (int p = o->n_pulses - 1; p >= 0; --p) {
#ifdef _OPENMP
#pragma omp parallel for num_threads(threads) schedule(dynamic, 1) if (threads > 1)
#endif
        for (int r = 0; r < o->ndom; ++r) {
            const size_t t = (size_t)p * o->ndom + r;
            const int32_t* m = o->maps + o->t_map_off[t];
            const int64_t S = o->t_size[t];
            float* dst = f + 3 * o->dom_offset[r];
            const float* src = f + 3 * (o->dom_offset[o->t_recv[t]] + o->t_off[t]);
            for (int64_t i = 0; i < S; ++i) {
                dst[3 * (int64_t)m[i] + 0] += src[3 * i + 0];
                dst[3 * (int64_t)m[i] + 1] += src[3 * i + 1];
                dst[3 * (int64_t)m[i] + 2] += src[3 * i + 2];
            }
        }
    }
}

void oracle_exchange_coords(const oracle_dd* o, float* x) { exchange_coords_impl(o, x, 1); }
void oracle_exchange_forces(const oracle_dd* o, float* f) { exchange_forces_impl(o, f, 1); }

/* The same exchanges with the senders of each pulse spread over `threads`
 * OpenMP threads (clamped to at least 1). Without OpenMP support at compile
 * time they run on one thread; oracle_max_threads() then returns 1. */
void oracle_exchange_coords_par(const oracle_dd* o, float* x, int threads) {
    exchange_coords_impl(o, x, threads < 1 ? 1 : threads);
}
void oracle_exchange_forces_par(const oracle_dd* o, float* f, int threads) {
    exchange_forces_impl(o, f, threads < 1 ? 1 : threads);
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
