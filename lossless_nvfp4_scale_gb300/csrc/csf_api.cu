// Host side of the CSF C ABI declared in include/csf.h: argument checks,
// launch configuration and dispatch.  Every step of the codec runs in the
// kernels of csf_decode.cu and csf_prepare.cu; nothing here touches the data.
#include <cstring>
#include <mutex>

#include "csf_internal.cuh"

using namespace csfk;

namespace csfk {

csf_status check_geometry(const csf_geometry *g, uint64_t *n, uint64_t *rows) {
    if (!g) return CSF_ERR_ARG;
    if (g->kind != CSF_NVFP4 && g->kind != CSF_MXFP4) return CSF_ERR_ARG;
    if (g->num_experts < 1 || g->rows < 1 || g->cols < 1) return CSF_ERR_ARG;
    const uint64_t r = (uint64_t)g->num_experts * (uint64_t)g->rows;
    const uint64_t e = r * (uint64_t)g->cols;
    if (r >= (1ull << 31) || e >= (1ull << 40) || g->cols >= (1 << 24)) return CSF_ERR_UNSUPPORTED;
    *n = e;
    *rows = r;
    return CSF_OK;
}

static bool is_aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

csf_status prepare_check(const uint8_t *dense, const csf_stack *out, uint64_t exc_capacity, PrepPlan *plan) {
    if (!dense || !out) return CSF_ERR_ARG;
    csf_status st = check_geometry(&out->g, &plan->n, &plan->rows);
    if (st != CSF_OK) return st;
    const csf_geometry &g = out->g;
    if (!out->base || !out->offsets || !out->exc_index || !is_aligned16(out->offsets)) return CSF_ERR_ARG;
    if (g.kind == CSF_MXFP4 && (!out->escapes || !is_aligned16(out->escapes))) return CSF_ERR_ARG;
    if (exc_capacity > 0 && !out->exc_bytes) return CSF_ERR_ARG;
    if (g.cols >= 65536) return CSF_ERR_UNSUPPORTED;
    const int32_t tr = prepare_tile_rows(g.kind, g.cols);
    if ((uint64_t)tr * g.cols >= (1ull << 24)) return CSF_ERR_UNSUPPORTED;
    plan->scratch_bytes = 16 + 8 * ((plan->rows + tr - 1) / tr);
    plan->fused_bytes = prepare_fused_scratch_bytes(g.kind, g.cols, plan->rows);
    plan->fused = false;
    plan->staged = true;
    plan->smem = 0;
    return CSF_OK;
}

csf_status prepare_configure(const uint8_t *dense, const csf_geometry &g, PrepPlan *plan) {
    const int32_t tr = prepare_tile_rows(g.kind, g.cols);
    plan->staged = prepare_stages_rows(g.kind, g.cols, dense);
    plan->smem = prepare_smem_bytes(g.kind, g.cols, tr, plan->staged);
    if (plan->smem > 200 * 1024) return CSF_ERR_UNSUPPORTED;
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, dense) != cudaSuccess) {
        cudaGetLastError();
        return CSF_ERR_ARG;
    }
    if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged) return CSF_ERR_ARG;
    return CSF_OK;
}

csf_status prepare_enqueue(const uint8_t *dense, const csf_stack &out, uint64_t exc_capacity, void *scratch,
                           const PrepPlan &plan, cudaStream_t s) {
    if (prepare_needs_cleared_scratch(out.g.cols) &&
        cudaMemsetAsync(scratch, 0, plan.scratch_bytes, s) != cudaSuccess) {   // ticket and status words start at 0
        cudaGetLastError();
        return CSF_ERR_CUDA;
    }
    PrepParams p;
    make_prep_params(p, dense, out, exc_capacity, scratch, plan.rows, plan.n, plan.staged, plan.fused);
    if (launch_prepare(p, plan.smem, s) != cudaSuccess) {
        cudaGetLastError();
        return CSF_ERR_CUDA;
    }
    return CSF_OK;
}

}  // namespace csfk

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    bool init = false;
    int sms = 0;
    int occ_full[3] = {0, 0, 0};   // full-stack decode, per DecodeKinds
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];

csf_status device_info(DeviceInfo *out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return CSF_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceInfo &d = g_dev[dev];
    if (!d.init) {
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return CSF_ERR_CUDA;
        }
        for (int k = 0; k < 3; ++k) {
            if (decode_occupancy(false, k, 0, &d.occ_full[k]) != cudaSuccess) {
                cudaGetLastError();
                return CSF_ERR_CUDA;
            }
            if (d.occ_full[k] < 1) d.occ_full[k] = 1;
        }
        d.init = true;
    }
    *out = d;
    return CSF_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

uint64_t round16(uint64_t v) { return (v + 15) & ~15ull; }

csf_status geometry(const csf_geometry *g, uint64_t *n, uint64_t *rows) { return check_geometry(g, n, rows); }

// Scratch of a prepare.  Rows of up to 255 bytes, up to 1 M of them: the
// fused path's per-tile totals and exception slots (about the dense size).
// Otherwise 16 bytes and one 8-byte word per tile of rows (per-tile totals
// of the two-kernel path, or a ticket counter and look-back words).
uint64_t prepare_scratch_bytes(const csf_geometry *g, uint64_t rows) {
    const uint64_t fused = prepare_fused_scratch_bytes(g->kind, g->cols, rows);
    if (fused) return fused;
    const int32_t tr = prepare_tile_rows(g->kind, g->cols);
    const uint64_t tiles = (rows + tr - 1) / tr;
    return 16 + 8 * tiles;
}

int ws_alignment(const void *p) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    if ((a & 31) == 0) return 32;
    if ((a & 15) == 0) return 16;
    if ((a & 3) == 0) return 4;
    return 1;
}

csf_status fill_stack(const csf_stack *s, uint8_t *ws, size_t ws_bytes, DecStack *d) {
    if (!s || !ws) return CSF_ERR_ARG;
    uint64_t n = 0, rows = 0;
    csf_status st = geometry(&s->g, &n, &rows);
    if (st != CSF_OK) return st;
    if (!s->base || !s->offsets || !s->exc_index || !aligned16(s->offsets)) return CSF_ERR_ARG;
    if (s->g.kind == CSF_MXFP4 && (!s->escapes || !aligned16(s->escapes))) return CSF_ERR_ARG;
    if (s->num_exc > 0 && !s->exc_bytes) return CSF_ERR_ARG;
    if (s->num_exc > 0xFFFFFFFFull) return CSF_ERR_ARG;
    if (ws_bytes < n) return CSF_ERR_SIZE;
    const int chunk = s->g.kind == CSF_NVFP4 ? kLaneNv : kLaneMx;
    std::memset(d, 0, sizeof *d);
    d->base = s->base;
    d->offsets = s->offsets;
    d->escapes = s->escapes;
    d->exc_index = s->exc_index;
    d->exc_bytes = s->exc_bytes;
    d->ws = ws;
    d->err = s->error_word;
    d->num_exc = s->num_exc;
    d->rows = rows;
    d->n = n;
    d->R = s->g.rows;
    d->C = s->g.cols;
    d->kind = s->g.kind;
    d->rb = unit_rows(s->g.cols, chunk);
    const uint32_t step_el = 32u * (uint32_t)chunk;
    d->step_r = step_el / (uint32_t)s->g.cols;
    d->step_q = step_el % (uint32_t)s->g.cols;
    d->ws_align = ws_alignment(ws);
    d->off_align32 = (reinterpret_cast<uintptr_t>(s->offsets) & 31u) == 0 ? 1 : 0;
    d->off_bytes = s->g.kind == CSF_NVFP4 ? round16((n + 1) / 2) : round16((n + 7) / 8);
    d->max_units = (1ull << 30) / ((uint64_t)d->rb * (uint64_t)d->C);
    if (d->max_units < 1) d->max_units = 1;
    return CSF_OK;
}

uint64_t blocked_bytes(const csf_geometry *g) {
    const uint64_t RP = ((uint64_t)g->rows + kTileRows - 1) / kTileRows * kTileRows;
    const uint64_t CP = ((uint64_t)g->cols + 3) / 4 * 4;
    return (uint64_t)g->num_experts * RP * CP;
}

uint64_t units_full(const DecStack &d) { return (d.rows + d.rb - 1) / d.rb; }

uint64_t units_all_experts(const DecStack &d, int E) {
    // Upper bound on the units of all experts' row ranges: each expert can
    // add one partial unit at each end.
    const uint64_t span = (uint64_t)E * (uint64_t)(d.r_hi - d.r_lo);
    return (span + d.rb - 1) / d.rb + 2ull * (uint64_t)E;
}

// A checked decode launch: parameters, grid and shared memory.  Building it
// has no side effect, so callers can enqueue stream waits only once the
// arguments are known to be good.
struct DecodeLaunch {
    DecParams p;
    size_t smem;
    int grid;
    bool per_expert;
    bool blocked;
    bool buffered;
};

#ifndef CSF_BLOCKS_MAX_COLS
#define CSF_BLOCKS_MAX_COLS 256
#endif
constexpr int32_t kBlocksMaxCols = CSF_BLOCKS_MAX_COLS;


csf_status plan_decode(const csf_decode_part *parts, int nparts, const void *expert_start, int es64,
                       DecodeLaunch *L) {
    if (!parts || nparts < 1 || nparts > 2) return CSF_ERR_ARG;
    DecParams &p = L->p;
    std::memset(&p, 0, sizeof p);
    bool whole = true;
    const int32_t layout = parts[0].layout;
    if (layout != CSF_LAYOUT_ROWS && layout != CSF_LAYOUT_BLOCKED) return CSF_ERR_ARG;
    const bool blocked = layout == CSF_LAYOUT_BLOCKED;
    for (int i = 0; i < nparts; ++i) {
        const csf_decode_part &q = parts[i];
        if (q.layout != layout) return CSF_ERR_ARG;
        csf_status st = fill_stack(q.stack, q.ws, q.ws_bytes, &p.st[i]);
        if (st != CSF_OK) return st;
        if (q.row_lo < 0 || q.row_lo >= q.row_hi || q.row_hi > q.stack->g.rows) return CSF_ERR_ARG;
        if (blocked) {
            if (!aligned16(q.ws)) return CSF_ERR_ARG;
            if (q.row_lo % kTileRows != 0 || (q.row_hi % kTileRows != 0 && q.row_hi != q.stack->g.rows))
                return CSF_ERR_ARG;
            if (q.ws_bytes < blocked_bytes(&q.stack->g)) return CSF_ERR_SIZE;
        }
        p.st[i].r_lo = q.row_lo;
        p.st[i].r_hi = q.row_hi;
        const int32_t rb = p.st[i].rb;
        if (q.stack->g.rows % rb == 0)
            p.st[i].upe = (uint32_t)((q.row_hi + rb - 1) / rb - q.row_lo / rb);
        if (q.row_lo != 0 || q.row_hi != q.stack->g.rows) whole = false;
        if (q.stack->g.num_experts != parts[0].stack->g.num_experts) return CSF_ERR_ARG;
    }
    p.nstacks = nparts;
    p.uniform = 1;
    for (int i = 0; i < nparts; ++i)
        if (p.st[i].upe == 0) p.uniform = 0;
    p.E = parts[0].stack->g.num_experts;
    p.expert_start = expert_start;
    p.es64 = es64 ? 1 : 0;
    const bool per_expert = expert_start != nullptr || !whole;
    if (blocked ? expert_start != nullptr : per_expert)
        if (p.E > kMaxRoutedExperts) return CSF_ERR_UNSUPPORTED;

    DeviceInfo di;
    csf_status st = device_info(&di);
    if (st != CSF_OK) return st;
    L->blocked = blocked;
    L->buffered = false;
    if (blocked) {
        // Work per 128-row block of an expert; the routed active list in
        // dynamic shared memory.  Rows up to kBlocksMaxCols bytes: one thread
        // block per 128-row block, decoded into its shared-memory buffer
        // (decode_blocks_kernel).  Wider rows: one warp per 128-row block,
        // line by line in registers (decode_tiles_kernel).
        int32_t cmax = 0;
        for (int i = 0; i < nparts; ++i)
            if (p.st[i].C > cmax) cmax = p.st[i].C;
        const size_t act = expert_start ? (4ull * (uint64_t)p.E + 15) & ~(size_t)15 : 0;
        L->buffered = cmax <= kBlocksMaxCols;
        size_t smem = act;
        if (L->buffered) {
            p.buf_off = (uint32_t)act;
            p.buf_bytes = (uint32_t)(((size_t)kTileRows * (size_t)cmax + 32 + 15) & ~(size_t)15);
            smem += p.buf_bytes;
        }
        int occ = 0;
        const cudaError_t oe = L->buffered ? decode_blocks_occupancy(p, smem, &occ) : decode_tiles_occupancy(smem, &occ);
        if (oe != cudaSuccess) {
            cudaGetLastError();
            return CSF_ERR_CUDA;
        }
        if (occ < 1) return CSF_ERR_UNSUPPORTED;
        uint64_t items = 0;
        for (int i = 0; i < nparts; ++i)
            items += (uint64_t)p.E * (((uint64_t)(p.st[i].r_hi - p.st[i].r_lo) + kTileRows - 1) / kTileRows);
        uint64_t grid = (uint64_t)di.sms * (uint64_t)occ;
        const uint64_t per_block = L->buffered ? 1 : kTileBlockWarps;   // 128-row blocks per thread block
        const uint64_t need = (items + per_block - 1) / per_block;
        if (need < grid) grid = need;
        if (grid < 1) grid = 1;
        L->smem = smem;
        L->grid = (int)grid;
        L->per_expert = true;
        return CSF_OK;
    }
    size_t smem = 0;
    const int kinds = decode_kinds(p);
    int occ = di.occ_full[kinds];
    uint64_t units = 0;
    if (per_expert) {
        // Active list (E words); prefix arrays (2 x (E+1) words) unless uniform.
        smem = p.uniform ? (expert_start ? 4ull * (uint64_t)p.E : 0)
                         : 4ull * ((uint64_t)p.E + 2ull * ((uint64_t)p.E + 1));
        if (decode_occupancy(true, kinds, smem, &occ) != cudaSuccess) {
            cudaGetLastError();
            return CSF_ERR_CUDA;
        }
        if (occ < 1) occ = 1;
        for (int i = 0; i < nparts; ++i) units += units_all_experts(p.st[i], p.E);
    } else {
        for (int i = 0; i < nparts; ++i) units += units_full(p.st[i]);
    }
    uint64_t grid = (uint64_t)di.sms * (uint64_t)occ;
    const uint64_t need = (units + kWarps - 1) / kWarps;
    if (need < grid) grid = need;
    if (grid < 1) grid = 1;
    L->smem = smem;
    L->grid = (int)grid;
    L->per_expert = per_expert;
    return CSF_OK;
}

csf_status launch(const DecodeLaunch &L, void *stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const cudaError_t e = !L.blocked     ? launch_decode(L.p, L.grid, L.smem, L.per_expert, st)
                          : L.buffered ? launch_decode_blocks(L.p, L.grid, L.smem, st)
                                          : launch_decode_tiles(L.p, L.grid, L.smem, st);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return CSF_ERR_CUDA;
    }
    return CSF_OK;
}

csf_status run_decode(const csf_decode_part *parts, int nparts, const void *expert_start, int es64,
                      void *stream) {
    DecodeLaunch L;
    csf_status st = plan_decode(parts, nparts, expert_start, es64, &L);
    if (st != CSF_OK) return st;
    return launch(L, stream);
}

csf_decode_part whole_part(const csf_stack *s, uint8_t *ws, size_t ws_bytes) {
    csf_decode_part q;
    q.stack = s;
    q.ws = ws;
    q.ws_bytes = ws_bytes;
    q.row_lo = 0;
    q.row_hi = s ? s->g.rows : 0;
    q.layout = CSF_LAYOUT_ROWS;
    return q;
}

}  // namespace

extern "C" {

const char *csf_status_string(csf_status status) {
    switch (status) {
    case CSF_OK: return "ok";
    case CSF_ERR_ARG: return "invalid argument";
    case CSF_ERR_SIZE: return "buffer too small";
    case CSF_ERR_UNSUPPORTED: return "unsupported geometry";
    case CSF_ERR_CUDA: return "CUDA error";
    }
    return "unknown status";
}

int csf_abi_version(void) { return CSF_ABI_VERSION; }

csf_status csf_sizes(const csf_geometry *g, csf_sizes_t *out) {
    if (!out) return CSF_ERR_ARG;
    uint64_t n = 0, rows = 0;
    csf_status st = geometry(g, &n, &rows);
    if (st != CSF_OK) return st;
    out->dense = n;
    out->base = rows;
    if (g->kind == CSF_NVFP4) {
        out->offsets = round16((n + 1) / 2);
        out->escapes = 0;
    } else {
        out->offsets = round16((n + 7) / 8);
        out->escapes = round16((n + 7) / 8);
    }
    out->exc_index = 4 * (rows + 1);
    out->prepare_scratch = prepare_scratch_bytes(g, rows);
    out->blocked = blocked_bytes(g);
    const uint64_t nrb = ((uint64_t)g->rows + kTileRows - 1) / kTileRows, ncb = ((uint64_t)g->cols + 3) / 4;
    const uint64_t tiles = (uint64_t)g->num_experts * nrb * ncb;
    out->tiled_codes = tiles * (g->kind == CSF_NVFP4 ? 256u : 128u);
    out->tiled_bases = (uint64_t)g->num_experts * nrb * 128u;
    out->tiled_index = 4 * (tiles + 1);
    return CSF_OK;
}

csf_status csf_prepare(const uint8_t *dense, csf_stack *out, uint64_t exc_capacity, void *scratch,
                       size_t scratch_bytes, void *stream) {
    if (!scratch) return CSF_ERR_ARG;
    PrepPlan plan;
    csf_status st = prepare_check(dense, out, exc_capacity, &plan);
    if (st != CSF_OK) return st;
    if ((reinterpret_cast<uintptr_t>(scratch) & 7u) != 0) return CSF_ERR_ARG;
    if (scratch_bytes < plan.scratch_bytes) return CSF_ERR_SIZE;
    plan.fused = plan.fused_bytes != 0 && scratch_bytes >= plan.fused_bytes;
    st = prepare_configure(dense, out->g, &plan);
    if (st != CSF_OK) return st;
    return prepare_enqueue(dense, *out, exc_capacity, scratch, plan, static_cast<cudaStream_t>(stream));
}

csf_status csf_decode(const csf_stack *s, uint8_t *ws, size_t ws_bytes, const void *expert_start,
                      int expert_start_is_int64, void *stream) {
    if (!s) return CSF_ERR_ARG;
    const csf_decode_part q = whole_part(s, ws, ws_bytes);
    return run_decode(&q, 1, expert_start, expert_start_is_int64, stream);
}

csf_status csf_decode_pair(const csf_stack *gate, uint8_t *gate_ws, size_t gate_ws_bytes, const csf_stack *down,
                           uint8_t *down_ws, size_t down_ws_bytes, const void *expert_start,
                           int expert_start_is_int64, void *stream) {
    if (!gate || !down) return CSF_ERR_ARG;
    const csf_decode_part q[2] = {whole_part(gate, gate_ws, gate_ws_bytes), whole_part(down, down_ws, down_ws_bytes)};
    return run_decode(q, 2, expert_start, expert_start_is_int64, stream);
}

csf_status csf_decode_rows(const csf_decode_part *parts, int num_parts, const void *expert_start,
                           int expert_start_is_int64, void *stream) {
    if (!parts || num_parts < 1 || num_parts > 2) return CSF_ERR_ARG;
    for (int i = 0; i < num_parts; ++i)
        if (!parts[i].stack) return CSF_ERR_ARG;
    return run_decode(parts, num_parts, expert_start, expert_start_is_int64, stream);
}

csf_status csf_expand(const csf_decode_part *parts, int num_parts, void *after, void *done, void *stream) {
    if (!parts || num_parts < 1 || num_parts > 2) return CSF_ERR_ARG;
    for (int i = 0; i < num_parts; ++i)
        if (!parts[i].stack) return CSF_ERR_ARG;
    DecodeLaunch L;
    csf_status st = plan_decode(parts, num_parts, nullptr, 0, &L);
    if (st != CSF_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (after && cudaStreamWaitEvent(s, static_cast<cudaEvent_t>(after), 0) != cudaSuccess) {
        cudaGetLastError();
        return CSF_ERR_CUDA;
    }
    st = launch(L, stream);
    if (st != CSF_OK) return st;
    if (done && cudaEventRecord(static_cast<cudaEvent_t>(done), s) != cudaSuccess) {
        cudaGetLastError();
        return CSF_ERR_CUDA;
    }
    return CSF_OK;
}

csf_status csf_tiled_pack(const csf_stack *src, csf_tiled *dst, uint64_t exc_capacity, void *stream) {
    if (!src || !dst) return CSF_ERR_ARG;
    uint64_t n = 0, rows = 0;
    csf_status st = geometry(&src->g, &n, &rows);
    if (st != CSF_OK) return st;
    const csf_geometry &g = src->g;
    if (dst->g.kind != g.kind || dst->g.num_experts != g.num_experts || dst->g.rows != g.rows ||
        dst->g.cols != g.cols)
        return CSF_ERR_ARG;
    if (!dst->codes || !dst->bases || !dst->tile_index || !aligned16(dst->codes) || !aligned16(dst->bases))
        return CSF_ERR_ARG;
    if (exc_capacity > 0 && !dst->exc_bytes) return CSF_ERR_ARG;
    if (src->num_exc > 0xFFFFFFFFull) return CSF_ERR_UNSUPPORTED;
    // The source read through the decode's stack view (its workspace unused).
    DecStack S;
    uint8_t dummy = 0;
    st = fill_stack(src, &dummy, n, &S);
    if (st != CSF_OK) return st;
    S.err = dst->error_word;
    TiledOut O;
    O.codes = dst->codes;
    O.bases = dst->bases;
    O.tile_index = dst->tile_index;
    O.exc_bytes = dst->exc_bytes;
    O.exc_capacity = exc_capacity;
    O.err = dst->error_word;
    DeviceInfo di;
    st = device_info(&di);
    if (st != CSF_OK) return st;
    const uint64_t items = (uint64_t)g.num_experts * (((uint64_t)g.rows + kTileRows - 1) / kTileRows);
    uint64_t grid = (items + 3) / 4;                       // 4 warps a block, one (expert, row block) each
    const uint64_t cap = (uint64_t)di.sms * 16;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    if (launch_tiled_pack(S, O, (int)grid, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return CSF_ERR_CUDA;
    }
    return CSF_OK;
}

csf_status csf_tiled_decode(const csf_tiled *t, uint8_t *ws, size_t ws_bytes, const void *expert_start,
                            int expert_start_is_int64, void *stream) {
    if (!t || !ws) return CSF_ERR_ARG;
    uint64_t n = 0, rows = 0;
    csf_status st = geometry(&t->g, &n, &rows);
    if (st != CSF_OK) return st;
    const csf_geometry &g = t->g;
    if (!t->codes || !t->bases || !t->tile_index || !aligned16(t->codes) || !aligned16(t->bases) || !aligned16(ws))
        return CSF_ERR_ARG;
    if (t->num_exc > 0 && !t->exc_bytes) return CSF_ERR_ARG;
    if (t->num_exc > 0xFFFFFFFFull) return CSF_ERR_ARG;
    if (ws_bytes < blocked_bytes(&g)) return CSF_ERR_SIZE;
    if (expert_start && g.num_experts > kMaxRoutedExperts) return CSF_ERR_UNSUPPORTED;
    DecStack S;
    std::memset(&S, 0, sizeof S);
    S.ws = ws;
    S.err = t->error_word;
    S.rows = rows;
    S.n = n;
    S.R = g.rows;
    S.C = g.cols;
    S.kind = g.kind;
    TiledIn I;
    std::memset(&I, 0, sizeof I);
    I.codes = t->codes;
    I.bases = t->bases;
    I.tile_index = t->tile_index;
    I.exc_bytes = t->exc_bytes;
    I.num_exc = t->num_exc;
    I.expert_start = expert_start;
    I.es64 = expert_start_is_int64 ? 1 : 0;
    DeviceInfo di;
    st = device_info(&di);
    if (st != CSF_OK) return st;
    const size_t smem = expert_start ? 4ull * (uint64_t)g.num_experts : 0;
    int occ = 0;
    if (tiled_decode_occupancy(g.kind, smem, &occ) != cudaSuccess) {
        cudaGetLastError();
        return CSF_ERR_CUDA;
    }
    if (occ < 1) occ = 1;
    const uint64_t tiles = (uint64_t)g.num_experts * (((uint64_t)g.rows + kTileRows - 1) / kTileRows) *
                           (((uint64_t)g.cols + 3) / 4);
    uint64_t grid = (uint64_t)di.sms * (uint64_t)occ;
    const uint64_t need = (tiles + 3) / 4;
    if (need < grid) grid = need;
    if (grid < 1) grid = 1;
    if (launch_tiled_decode(S, I, (int)grid, smem, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return CSF_ERR_CUDA;
    }
    return CSF_OK;
}

csf_status csf_tiled_checksum(const csf_tiled *t, uint32_t *sums, size_t sums_count, const void *expert_start,
                              int expert_start_is_int64, void *stream) {
    if (!t || !sums) return CSF_ERR_ARG;
    uint64_t n = 0, rows = 0;
    csf_status st = geometry(&t->g, &n, &rows);
    if (st != CSF_OK) return st;
    const csf_geometry &g = t->g;
    if (!t->codes || !t->bases || !t->tile_index || !aligned16(t->codes) || !aligned16(t->bases)) return CSF_ERR_ARG;
    if (t->num_exc > 0 && !t->exc_bytes) return CSF_ERR_ARG;
    if (t->num_exc > 0xFFFFFFFFull) return CSF_ERR_ARG;
    const uint64_t tiles = (uint64_t)g.num_experts * (((uint64_t)g.rows + kTileRows - 1) / kTileRows) *
                           (((uint64_t)g.cols + 3) / 4);
    if (sums_count < tiles) return CSF_ERR_SIZE;
    if (expert_start && g.num_experts > kMaxRoutedExperts) return CSF_ERR_UNSUPPORTED;
    DecStack S;
    std::memset(&S, 0, sizeof S);
    S.err = t->error_word;
    S.rows = rows;
    S.n = n;
    S.R = g.rows;
    S.C = g.cols;
    S.kind = g.kind;
    TiledIn I;
    std::memset(&I, 0, sizeof I);
    I.codes = t->codes;
    I.bases = t->bases;
    I.tile_index = t->tile_index;
    I.exc_bytes = t->exc_bytes;
    I.num_exc = t->num_exc;
    I.expert_start = expert_start;
    I.es64 = expert_start_is_int64 ? 1 : 0;
    DeviceInfo di;
    st = device_info(&di);
    if (st != CSF_OK) return st;
    const size_t smem = expert_start ? 4ull * (uint64_t)g.num_experts : 0;
    int occ = 0;
    if (tiled_checksum_occupancy(g.kind, smem, &occ) != cudaSuccess) {
        cudaGetLastError();
        return CSF_ERR_CUDA;
    }
    if (occ < 1) occ = 1;
    uint64_t grid = (uint64_t)di.sms * (uint64_t)occ;
    const uint64_t need = (tiles + 3) / 4;
    if (need < grid) grid = need;
    if (grid < 1) grid = 1;
    if (launch_tiled_checksum(S, I, sums, (int)grid, smem, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return CSF_ERR_CUDA;
    }
    return CSF_OK;
}

csf_status csf_selftest_lookback_timeout(uint32_t *error_word) {
    if (!error_word) return CSF_ERR_ARG;
    *error_word = 0;
    // A 512 x 300 NVFP4 stack: rows wider than 255 bytes take the single-pass
    // kernel, whose tiles (48 rows) chain their exception counts through a
    // decoupled look-back.  The ticket counter starts at 1, so no block takes
    // tile 0 and the next tiles' look-backs wait on a status word that nothing
    // writes; with a short poll limit the waits give up.
    csf_stack st;
    std::memset(&st, 0, sizeof st);
    st.g.kind = CSF_NVFP4;
    st.g.num_experts = 1;
    st.g.rows = 512;
    st.g.cols = 300;
    const uint64_t rows = 512, n = 512 * 300;
    const int32_t tr = prepare_tile_rows(st.g.kind, st.g.cols);
    const size_t smem = prepare_smem_bytes(st.g.kind, st.g.cols, tr, false);
    const uint64_t need = prepare_scratch_bytes(&st.g, rows);
    auto up = [](size_t v) { return (v + 255) & ~(size_t)255; };
    // dense, base, offsets, index, exceptions, error word, scratch
    const size_t off_dense = 0, off_base = up(off_dense + n), off_offsets = up(off_base + rows),
                 off_index = up(off_offsets + n / 2), off_exc = up(off_index + 4 * (rows + 1)),
                 off_err = up(off_exc + n), off_scratch = up(off_err + 16);
    uint8_t *mem = nullptr;
    if (cudaMalloc(&mem, off_scratch + need) != cudaSuccess) {
        cudaGetLastError();
        return CSF_ERR_CUDA;
    }
    cudaStream_t s = nullptr;
    csf_status ret = CSF_OK;
    const uint32_t one = 1;
    PrepParams p;
    st.base = mem + off_base;
    st.offsets = mem + off_offsets;
    st.exc_index = reinterpret_cast<uint32_t *>(mem + off_index);
    st.exc_bytes = mem + off_exc;
    st.error_word = reinterpret_cast<uint32_t *>(mem + off_err);
    make_prep_params(p, mem + off_dense, st, n, mem + off_scratch, rows, n, false, false);
    p.spin_limit = 4096;
    if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess ||
        cudaMemsetAsync(mem, 0, off_scratch + need, s) != cudaSuccess ||
        cudaMemcpyAsync(mem + off_scratch, &one, sizeof one, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        launch_prepare(p, smem, s) != cudaSuccess ||
        cudaMemcpyAsync(error_word, st.error_word, sizeof *error_word, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        ret = CSF_ERR_CUDA;
    }
    if (s) cudaStreamDestroy(s);
    cudaFree(mem);
    return ret;
}

}  // extern "C"
