// Host side of libpkv: the C ABI declared in include/pkv.h.
//
// pkv_decode / pkv_step validate their arguments on the host, carve the
// caller's workspace, and enqueue three kernels on the caller's stream:
//   prep (QK-norm + RoPE + append) -> split-KV attention -> split combine.
// The second and third use programmatic dependent launch so their prologues
// overlap the tail of the kernel before them.  Nothing here allocates or
// synchronises on the call path.
#include <cudaTypedefs.h>

#include <algorithm>
#include <array>
#include <climits>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "pkv_internal.h"

namespace pkv {

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Workspace of one call: per token its attended length and table row (step
// mode), the prefix of pages over tokens, a validity flag per (token, kv head)
// unit, and one partial (4 heads x 128 fp32 + 4 log-sum-exps) per piece of a
// unit split between intervals of the attention's work split: unit u's piece in
// interval i sits at u + i, and there are at most C static slices plus
// kDynChunksPerCta * C chunks, so U + C (1 + kDynChunksPerCta) slots.
Plan make_plan(const pkv_pool* pool, int tokens, int pages, int prompt_tokens)
{
    Plan pl;
    pl.tokens = tokens;
    pl.pages = pages;
    pl.ctas = pool->ctas_override > 0 ? pool->ctas_override : pool->ctas_per_sm * pool->num_sms;
    const size_t G = (size_t)pool->cfg.kv_heads;
    const size_t units = (size_t)tokens * G;
    const size_t slots = units + (size_t)pl.ctas * (1 + kDynChunksPerCta);
    size_t off = 0;
    pl.off_len = off;
    off = align_up(off + sizeof(int32_t) * tokens, 256);
    pl.off_row = off;
    off = align_up(off + sizeof(int32_t) * tokens, 256);
    pl.off_prefix = off;
    off = align_up(off + sizeof(int32_t) * (tokens + 2), 256);
    pl.off_unit_ok = off;
    off = align_up(off + sizeof(int32_t) * units, 256);
    pl.off_po = off;
    off = align_up(off + sizeof(float) * slots * kGroup * kHeadDim, 256);
    pl.off_plse = off;
    off = align_up(off + sizeof(float) * slots * kGroup, 256);
    pl.off_sched = off;
    off = align_up(off + sizeof(int32_t), 256);
    pl.off_qhat = off;
    off = align_up(off + (size_t)prompt_tokens * pool->cfg.heads * kHeadDim * 2, 256);
    pl.total = off;
    pl.claim = nullptr;
    return pl;
}

// decode:  attention (which also validates rows and appends their k/v) -> combine.
// step:    prep (validates every token, appends every k/v) -> prompt-token
//          attention on the tensor cores -> step-row attention -> combine.
// prefill: prep -> prompt-token attention.
// All but the first kernel use programmatic dependent launch: each is
// scheduled while the one before it drains and waits for it before touching
// memory.
int enqueue(pkv_pool* pool, const StepArgs& a, const Plan& plan, cudaStream_t s)
{
    const bool decode = a.P == 0;
    const bool timed = pool->timer_on != 0;
    const int slot = timed ? (int)(pool->timer_count.fetch_add(1) % kTimerSlots) : 0;
    if (!decode && a.steps == 0) {  // prompts only: prep -> prompt-token attention (the timed kernel)
        if (launch_prep(pool, a, plan, s) != cudaSuccess) return PKV_ECUDA;
        if (timed && cudaEventRecord(pool->ev_start[slot], s) != cudaSuccess) return PKV_ECUDA;
        if (launch_prefill(pool, a, plan, pool->num_sms, false, s) != cudaSuccess) return PKV_ECUDA;
        if (timed && cudaEventRecord(pool->ev_stop[slot], s) != cudaSuccess) return PKV_ECUDA;
        return PKV_OK;
    }
    StepArgs as = a;  // the tokens the attention + combine kernels see
    Plan ps = plan;
    ps.claim = pool->claims + (pool->call_seq++ % kClaimSlots);
    if (!decode) {
        if (launch_prep(pool, a, plan, s) != cudaSuccess) return PKV_ECUDA;
        // beside the step rows' attention (programmatic launch), the prompt attention keeps
        // part of the SMs and leaves the rest to it (prompt_sms); timed calls run them in turn
        if (launch_prefill(pool, a, plan, pool->num_sms, !timed, s) != cudaSuccess) return PKV_ECUDA;
        // the step rows are tokens P..P+rows-1
        const size_t qrow = (size_t)pool->cfg.heads * pool->cfg.head_dim * 2;
        as.q = static_cast<const char*>(a.q) + (size_t)a.P * qrow;
        as.out = static_cast<char*>(a.out) + (size_t)a.P * qrow;
        ps.tokens = a.steps;
        ps.off_len += sizeof(int32_t) * a.P;
        ps.off_row += sizeof(int32_t) * a.P;
    }
    if (timed && cudaEventRecord(pool->ev_start[slot], s) != cudaSuccess) return PKV_ECUDA;
    if (launch_attn(pool, as, ps, decode, !timed, s) != cudaSuccess) return PKV_ECUDA;
    if (timed && cudaEventRecord(pool->ev_stop[slot], s) != cudaSuccess) return PKV_ECUDA;
    if (launch_combine(pool, as, ps, decode, s) != cudaSuccess) {
        // the combine resets this call's chunk counter; without it, reset it here
        cudaMemsetAsync(ps.claim, 0, sizeof(uint32_t), s);
        return PKV_ECUDA;
    }
    return PKV_OK;
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }
    return fn;
}

// 3-D tiled view {head_dim, num_slots, kv_heads} of one pool tensor; a box is
// 64 head-dim elements (128 bytes, the swizzle span) x 64 slots (one page).
static bool make_tmap(CUtensorMap* map, void* base, int64_t num_slots, int kv_heads)
{
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)kHeadDim, (cuuint64_t)num_slots, (cuuint64_t)kv_heads};
    cuuint64_t strides[2] = {(cuuint64_t)kHeadDim * 2, (cuuint64_t)num_slots * kHeadDim * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)kPageSize, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 2-D tiled view {inner, outer} of a row-major bf16 matrix with `row_bytes`
// between rows; a box is box_inner x box_outer elements with 128-byte swizzle,
// and reads past the matrix's edge fill zeros.
bool make_tmap_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                  uint32_t box_inner, uint32_t box_outer)
{
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
    cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool make_tmap_heads(CUtensorMap* map, const void* base, int heads, int tokens)
{
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)kHeadDim, (cuuint64_t)heads, (cuuint64_t)tokens};
    cuuint64_t strides[2] = {(cuuint64_t)kHeadDim * 2, (cuuint64_t)heads * kHeadDim * 2};
    cuuint32_t box[3] = {64, 1, 32};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

static int check_config(const pkv_config* c)
{
    if (c->heads <= 0 || c->kv_heads <= 0 || c->head_dim <= 0 || c->page_size <= 0 || c->max_seq <= 0)
        return PKV_EINVAL;
    if (c->heads % c->kv_heads != 0 || c->head_dim % 2 != 0) return PKV_EINVAL;
    if (!(c->rope_theta > 0.0) || !(c->eps >= 0.0) || !std::isfinite(c->rope_theta) || !std::isfinite(c->eps))
        return PKV_EINVAL;
    if (c->head_dim != kHeadDim || c->page_size != kPageSize || c->heads != kGroup * c->kv_heads)
        return PKV_ENOTIMPL;
    if (c->max_seq > (1 << 20) || c->kv_heads > 256) return PKV_ERANGE;
    if (c->rotary_dim < 0 || c->rotary_dim > c->head_dim || c->rotary_dim % 2) return PKV_EINVAL;
    if (c->rotary_dim % 32) return PKV_ENOTIMPL;
    return PKV_OK;
}

// RoPE tables: (cos, sin) of pos * theta^(-2i/head_dim), i < head_dim/2, for
// every position < max_seq, computed in double (qwen3-8b Nest files,
// src/rope.linnet tables; the pages evaluate the angle in f32, which at
// position 40959 is off by up to ~2e-3 rad) and kept as two fp32 tables: hi,
// the nearest fp32 values (q uses these), and lo, the remainders (k uses
// hi + lo, so its rotation keeps the double table's accuracy).
// (cos, sin) of pos * theta^(-2i/R) for i < R/2 (R = rotary dims), in double,
// kept as the nearest fp32 pair plus the fp32 of the remainder; entries past
// R/2 (partial rotation) are the identity (1, 0).
static void rope_tables(const pkv_config& c, std::vector<float2>& hi, std::vector<float2>& lo)
{
    const int half = c.head_dim / 2, R = c.rotary_dim > 0 ? c.rotary_dim : c.head_dim, rhalf = R / 2;
    hi.assign((size_t)c.max_seq * half, make_float2(1.f, 0.f));
    lo.assign((size_t)c.max_seq * half, make_float2(0.f, 0.f));
    std::vector<double> inv(rhalf);
    for (int i = 0; i < rhalf; ++i) inv[i] = std::pow(c.rope_theta, -2.0 * i / (double)R);
    for (int p = 0; p < c.max_seq; ++p)
        for (int i = 0; i < rhalf; ++i) {
            const double a = (double)p * inv[i];
            const double cs = std::cos(a), sn = std::sin(a);
            const float ch = (float)cs, sh = (float)sn;
            hi[(size_t)p * half + i] = make_float2(ch, sh);
            lo[(size_t)p * half + i] = make_float2((float)(cs - (double)ch), (float)(sn - (double)sh));
        }
}

static int create_pool(const pkv_config* cfg, int num_pages, void* k, void* v, bool owns, void* stream,
                       pkv_pool** out)
{
    if (!cfg || !out || num_pages <= 0) return PKV_EINVAL;
    *out = nullptr;
    int rc = check_config(cfg);
    if (rc != PKV_OK) return rc;
    const int64_t num_slots = (int64_t)num_pages * cfg->page_size;
    if (num_slots >= (int64_t(1) << 31)) return PKV_ERANGE;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PKV_EDEVICE;
    int major = 0, sms = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (major < 10 || sms <= 0) return PKV_EDEVICE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    pkv_pool* p = new (std::nothrow) pkv_pool();
    if (!p) return PKV_ENOMEM;
    p->cfg = *cfg;
    p->device = dev;
    p->num_sms = sms;
    p->num_pages = num_pages;
    p->num_slots = num_slots;
    p->owns_kv = owns;
    p->wait_ns = 1000000000ull;
    const size_t kv_bytes = (size_t)cfg->kv_heads * num_slots * cfg->head_dim * 2;
    const size_t tab = (size_t)cfg->max_seq * (cfg->head_dim / 2) * sizeof(float2);
    bool fail = false;
    if (owns) {
        fail |= cudaMalloc(&p->k, kv_bytes) != cudaSuccess;
        fail |= !fail && cudaMalloc(&p->v, kv_bytes) != cudaSuccess;
    } else {
        p->k = k;
        p->v = v;
    }
    fail |= !fail && cudaMalloc(reinterpret_cast<void**>(&p->rope_hi), tab) != cudaSuccess;
    fail |= !fail && cudaMalloc(reinterpret_cast<void**>(&p->rope_lo), tab) != cudaSuccess;
    fail |= !fail && cudaMalloc(reinterpret_cast<void**>(&p->err), 256) != cudaSuccess;
    if (fail) {
        cudaGetLastError();
        pkv_pool_free(p);
        return PKV_ENOMEM;
    }
    p->claims = p->err + 32;
    static_assert(32 + kClaimSlots <= 256 / 4, "the claim counters share the error word's allocation");
    std::vector<float2> rhi, rlo;
    rope_tables(*cfg, rhi, rlo);
    bool ok = true;
    if (owns) {
        ok &= cudaMemsetAsync(p->k, 0, kv_bytes, s) == cudaSuccess;
        ok &= cudaMemsetAsync(p->v, 0, kv_bytes, s) == cudaSuccess;
    }
    ok &= cudaMemcpyAsync(p->rope_hi, rhi.data(), tab, cudaMemcpyHostToDevice, s) == cudaSuccess;
    ok &= cudaMemcpyAsync(p->rope_lo, rlo.data(), tab, cudaMemcpyHostToDevice, s) == cudaSuccess;
    ok &= cudaMemsetAsync(p->err, 0, 256, s) == cudaSuccess;
    ok &= cudaStreamSynchronize(s) == cudaSuccess;  // the host vectors die with this call
    ok &= make_tmap(&p->tmap_k, p->k, num_slots, cfg->kv_heads);
    ok &= make_tmap(&p->tmap_v, p->v, num_slots, cfg->kv_heads);
    ok &= configure_kernels() == cudaSuccess;
    ok &= configure_prefill() == cudaSuccess;
    p->ctas_per_sm = attn_ctas_per_sm();
    ok &= p->ctas_per_sm > 0;
    if (!ok) {
        cudaGetLastError();
        pkv_pool_free(p);
        return PKV_ECUDA;
    }
    *out = p;
    return PKV_OK;
}

static bool aligned(const void* ptr, size_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) == 0; }

// ---- optional host pre-check (environment variable PKV_CHECK=1) ----------------------------
bool check_enabled()
{
    const char* e = std::getenv("PKV_CHECK");
    return e && e[0] == '1' && e[1] == 0;
}

// Copies the call's token tables to the host (synchronising the stream first)
// and rejects, with PKV_EINVAL, a call whose written slots are not distinct
// outside pool page 0, whose given prompt slots differ from those the table
// derives, or -- decode only, where each row's write is ordered before its own
// reads but not before other rows' -- in which a row reads a slot another row
// of the call writes.  Tokens the device would skip (position, row or page out
// of range) take no part: the device checks report them.
int host_precheck(const pkv_pool* pool, const StepArgs& a, cudaStream_t s)
{
    if (cudaStreamSynchronize(s) != cudaSuccess) return PKV_ECUDA;
    auto fetch = [](const int32_t* src, size_t n, std::vector<int32_t>& dst) {
        dst.resize(n);
        return n == 0 || cudaMemcpy(dst.data(), src, n * sizeof(int32_t), cudaMemcpyDeviceToHost) == cudaSuccess;
    };
    std::vector<int32_t> pos, prow, slots, steps, table;
    bool ok = fetch(a.positions, a.P, pos) && fetch(a.prow, a.P, prow) && fetch(a.step_positions, a.steps, steps);
    if (a.slots) ok = ok && fetch(a.slots, a.P, slots);
    if (a.table) ok = ok && fetch(a.table, (size_t)a.rows * a.pages, table);
    if (!ok) return PKV_ECUDA;
    const int S = pool->cfg.page_size;
    auto page = [&](int row, int j) -> int64_t {
        return a.table ? (int64_t)table[(size_t)row * a.pages + j] : (int64_t)row * a.pages + j;
    };
    // the slot the table gives token (row, p), or -1 if the device would skip the token
    auto derive = [&](int row, int p) -> int64_t {
        if (row < 0 || row >= a.rows || p < 0 || p >= pool->cfg.max_seq || p >= a.pages * S) return -1;
        for (int j = 0; j <= p / S; ++j) {
            const int64_t id = page(row, j);
            if (id < 0 || id >= pool->num_pages) return -1;
        }
        return page(row, p / S) * S + p % S;
    };
    std::vector<int64_t> written;
    for (int t = 0; t < a.P; ++t) {
        const int64_t d = derive(prow[t], pos[t]);
        if (d < 0) continue;
        if (a.slots) {
            if (slots[t] < 0 || slots[t] >= pool->num_slots) continue;
            if (slots[t] != d) return PKV_EINVAL;
        }
        written.push_back(d);
    }
    for (int b = 0; b < a.steps; ++b) {
        if (steps[b] == -1) continue;
        const int64_t d = derive(b, steps[b]);
        if (d >= 0) written.push_back(d);
    }
    std::sort(written.begin(), written.end());
    for (size_t i = 1; i < written.size(); ++i)
        if (written[i] == written[i - 1] && written[i] >= S) return PKV_EINVAL;
    if (a.P == 0 && a.steps > 0 && !a.q_hat) {
        // decode: no row may read (position s <= its own) a slot another row writes.
        // (page id, row, offset in page) of every write, sorted by page id
        std::vector<std::array<int64_t, 3>> w;
        for (int b = 0; b < a.steps; ++b) {
            if (steps[b] == -1) continue;
            const int64_t d = derive(b, steps[b]);
            if (d >= 0) w.push_back({d / S, b, d % S});
        }
        std::sort(w.begin(), w.end());
        for (int b = 0; b < a.steps; ++b) {
            if (steps[b] == -1 || derive(b, steps[b]) < 0) continue;
            const int last = steps[b] / S;
            for (int j = 0; j <= last; ++j) {
                const int64_t id = page(b, j);
                const int64_t lim = j == last ? steps[b] % S : S - 1;  // offsets row b reads in this page
                auto it = std::lower_bound(w.begin(), w.end(), std::array<int64_t, 3>{id, INT64_MIN, INT64_MIN});
                for (; it != w.end() && (*it)[0] == id; ++it)
                    if ((*it)[1] != b && (*it)[2] <= lim) return PKV_EINVAL;
            }
        }
    }
    return PKV_OK;
}

static int run_step(pkv_pool* pool, const StepArgs& a, size_t ws_bytes, void* stream)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != pool->device) return PKV_EDEVICE;
    // contiguous rows (no table): every row's pages must be in the pool
    if (!a.table && (int64_t)a.rows * a.pages > pool->num_pages) return PKV_ERANGE;
    if (check_enabled()) {
        const int rc = host_precheck(pool, a, static_cast<cudaStream_t>(stream));
        if (rc != PKV_OK) return rc;
    }
    const Plan plan = make_plan(pool, a.P + a.steps, a.pages, a.P);
    if (!a.ws || ws_bytes < plan.total) return PKV_EWORKSPACE;
    return enqueue(pool, a, plan, static_cast<cudaStream_t>(stream));
}

}  // namespace pkv

using namespace pkv;

extern "C" {

int pkv_config_default(pkv_config* cfg)
{
    if (!cfg) return PKV_EINVAL;
    cfg->heads = 32;
    cfg->kv_heads = 8;
    cfg->head_dim = 128;
    cfg->page_size = 64;
    cfg->max_seq = 40960;
    cfg->rope_theta = 1.0e6;
    cfg->eps = 1.0e-6;
    cfg->rotary_dim = 128;
    return PKV_OK;
}

const char* pkv_strerror(int code)
{
    switch (code) {
        case PKV_OK: return "ok";
        case PKV_EINVAL: return "invalid argument";
        case PKV_ERANGE: return "size out of supported range";
        case PKV_ENOMEM: return "device allocation failed";
        case PKV_ECUDA: return "CUDA runtime error";
        case PKV_EWORKSPACE: return "workspace too small";
        case PKV_EDEVICE: return "no usable device or wrong device";
        case PKV_ENOTIMPL: return "configuration not supported by the kernels";
        default: return "unknown error";
    }
}

int pkv_pool_alloc(const pkv_config* cfg, int num_pages, void* stream, pkv_pool** out)
{
    return create_pool(cfg, num_pages, nullptr, nullptr, true, stream, out);
}

int pkv_pool_wrap(const pkv_config* cfg, int num_pages, void* k, void* v, void* stream, pkv_pool** out)
{
    if (!k || !v || !aligned(k, 256) || !aligned(v, 256)) return PKV_EINVAL;
    return create_pool(cfg, num_pages, k, v, false, stream, out);
}

int pkv_pool_free(pkv_pool* p)
{
    if (!p) return PKV_OK;
    int prev = -1;
    cudaGetDevice(&prev);
    cudaSetDevice(p->device);
    cudaDeviceSynchronize();
    if (p->owns_kv) {
        if (p->k) cudaFree(p->k);
        if (p->v) cudaFree(p->v);
    }
    if (p->rope_hi) cudaFree(p->rope_hi);
    if (p->rope_lo) cudaFree(p->rope_lo);
    if (p->err) cudaFree(p->err);
    if (p->ev_start) {
        for (int i = 0; i < kTimerSlots; ++i) {
            cudaEventDestroy(p->ev_start[i]);
            cudaEventDestroy(p->ev_stop[i]);
        }
        delete[] p->ev_start;
        delete[] p->ev_stop;
    }
    if (prev >= 0) cudaSetDevice(prev);
    delete p;
    return PKV_OK;
}

int pkv_pool_kv(const pkv_pool* pool, void** k, void** v, int64_t* num_slots)
{
    if (!pool) return PKV_EINVAL;
    if (k) *k = pool->k;
    if (v) *v = pool->v;
    if (num_slots) *num_slots = pool->num_slots;
    return PKV_OK;
}

int pkv_workspace_bytes(const pkv_pool* pool, int rows, int pages, int prefill_tokens, size_t* bytes)
{
    if (!pool || !bytes || rows < 0 || prefill_tokens < 0 || rows + prefill_tokens <= 0 || pages <= 0)
        return PKV_EINVAL;
    if ((int64_t)rows + prefill_tokens > (1 << 20) || (int64_t)rows * pages > INT32_MAX) return PKV_ERANGE;
    *bytes = make_plan(pool, rows + prefill_tokens, pages, prefill_tokens).total;
    return PKV_OK;
}

int pkv_decode(pkv_pool* pool, const void* q, const void* k, const void* v, const void* q_norm_w,
               const void* k_norm_w, const int32_t* positions, const int32_t* table, int rows, int pages,
               void* out, void* workspace, size_t workspace_bytes, void* stream)
{
    NvtxRange range("pkv_decode");
    if (!pool || !q || !k || !v || !q_norm_w || !k_norm_w || !positions || !out) return PKV_EINVAL;
    if (rows <= 0 || pages <= 0) return PKV_EINVAL;
    if (rows > (1 << 20) || (int64_t)rows * pages > INT32_MAX) return PKV_ERANGE;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 8) || !aligned(q_norm_w, 8) ||
        !aligned(k_norm_w, 8) || !aligned(positions, 4) || !aligned(table, 4))
        return PKV_EINVAL;
    if (workspace && !aligned(workspace, 256)) return PKV_EINVAL;
    StepArgs a = {q, k, v, q_norm_w, k_norm_w, nullptr, nullptr, nullptr, positions, table,
                  0, rows, pages, rows, out, static_cast<char*>(workspace)};
    return run_step(pool, a, workspace_bytes, stream);
}

int pkv_qkv_proj_append(pkv_pool* pool, const void* x, const void* w_qkv, int tokens, int hidden,
                        const void* q_norm_w, const void* k_norm_w, const int32_t* positions, const int32_t* table,
                        int pages, float* q_hat, void* stream)
{
    NvtxRange range("pkv_qkv_proj_append");
    if (!pool || !x || !w_qkv || !q_norm_w || !k_norm_w || !positions || !q_hat) return PKV_EINVAL;
    if (tokens <= 0 || hidden <= 0 || pages <= 0) return PKV_EINVAL;
    if (hidden % 64) return PKV_ENOTIMPL;
    if (tokens > (1 << 20) || hidden > (1 << 20) || (int64_t)tokens * pages > INT32_MAX) return PKV_ERANGE;
    if (!aligned(x, 16) || !aligned(w_qkv, 16) || !aligned(q_hat, 16) || !aligned(q_norm_w, 8) ||
        !aligned(k_norm_w, 8) || !aligned(positions, 4) || !aligned(table, 4))
        return PKV_EINVAL;
    if (!table && (int64_t)tokens * pages > pool->num_pages) return PKV_ERANGE;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != pool->device) return PKV_EDEVICE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (check_enabled()) {  // written slots must be distinct (the append is a scatter)
        const StepArgs a = {nullptr, nullptr, nullptr, q_norm_w, k_norm_w, nullptr, nullptr, nullptr, positions,
                            table, 0, tokens, pages, tokens, nullptr, nullptr, q_hat};
        const int rc = host_precheck(pool, a, s);
        if (rc != PKV_OK) return rc;
    }
    const QkvAppend fa = {q_norm_w, k_norm_w, positions, table, pages, q_hat};
    return launch_qkv_append(pool, x, w_qkv, tokens, hidden, fa, s) == cudaSuccess ? PKV_OK : PKV_ECUDA;
}

int pkv_decode_appended(pkv_pool* pool, const float* q_hat, const int32_t* positions, const int32_t* table, int rows,
                        int pages, void* out, void* workspace, size_t workspace_bytes, void* stream)
{
    NvtxRange range("pkv_decode_appended");
    if (!pool || !q_hat || !positions || !out) return PKV_EINVAL;
    if (rows <= 0 || pages <= 0) return PKV_EINVAL;
    if (rows > (1 << 20) || (int64_t)rows * pages > INT32_MAX) return PKV_ERANGE;
    if (!aligned(q_hat, 16) || !aligned(out, 8) || !aligned(positions, 4) || !aligned(table, 4)) return PKV_EINVAL;
    if (workspace && !aligned(workspace, 256)) return PKV_EINVAL;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != pool->device) return PKV_EDEVICE;
    if (!table && (int64_t)rows * pages > pool->num_pages) return PKV_ERANGE;
    const Plan plan = make_plan(pool, rows, pages, 0);
    if (!workspace || workspace_bytes < plan.total) return PKV_EWORKSPACE;
    const StepArgs a = {nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, positions, table,
                        0, rows, pages, rows, out, static_cast<char*>(workspace), q_hat};
    return enqueue(pool, a, plan, static_cast<cudaStream_t>(stream));
}

int pkv_step(pkv_pool* pool, const void* q, const void* k, const void* v, const void* q_norm_w,
             const void* k_norm_w, const int32_t* positions, const int32_t* prow, const int32_t* slots,
             const int32_t* step_positions, const int32_t* table, int P, int rows, int pages, void* out,
             void* workspace, size_t workspace_bytes, void* stream)
{
    NvtxRange range("pkv_step");
    if (!pool || !q || !k || !v || !q_norm_w || !k_norm_w || !positions || !prow || !step_positions || !out)
        return PKV_EINVAL;
    if (P <= 0 || rows <= 0 || pages <= 0) return PKV_EINVAL;
    if ((int64_t)P + rows > (1 << 20) || (int64_t)rows * pages > INT32_MAX) return PKV_ERANGE;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) || !aligned(q_norm_w, 8) ||
        !aligned(k_norm_w, 8) || !aligned(positions, 4) || !aligned(prow, 4) || !aligned(step_positions, 4) ||
        !aligned(table, 4) || (slots && !aligned(slots, 4)))
        return PKV_EINVAL;
    if (workspace && !aligned(workspace, 256)) return PKV_EINVAL;
    StepArgs a = {q, k, v, q_norm_w, k_norm_w, positions, prow, slots, step_positions, table,
                  P, rows, pages, rows, out, static_cast<char*>(workspace)};
    return run_step(pool, a, workspace_bytes, stream);
}

int pkv_prefill(pkv_pool* pool, const void* q, const void* k, const void* v, const void* q_norm_w,
                const void* k_norm_w, const int32_t* positions, const int32_t* prow, const int32_t* slots,
                const int32_t* table, int P, int rows, int pages, void* out, void* workspace,
                size_t workspace_bytes, void* stream)
{
    NvtxRange range("pkv_prefill");
    if (!pool || !q || !k || !v || !q_norm_w || !k_norm_w || !positions || !prow || !out) return PKV_EINVAL;
    if (P <= 0 || rows <= 0 || pages <= 0) return PKV_EINVAL;
    if (P > (1 << 20) || (int64_t)rows * pages > INT32_MAX) return PKV_ERANGE;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) || !aligned(q_norm_w, 8) ||
        !aligned(k_norm_w, 8) || !aligned(positions, 4) || !aligned(prow, 4) || !aligned(table, 4) ||
        (slots && !aligned(slots, 4)))
        return PKV_EINVAL;
    if (workspace && !aligned(workspace, 256)) return PKV_EINVAL;
    StepArgs a = {q, k, v, q_norm_w, k_norm_w, positions, prow, slots, nullptr, table,
                  P, rows, pages, 0, out, static_cast<char*>(workspace)};
    return run_step(pool, a, workspace_bytes, stream);
}

int pkv_linear_workspace_bytes(const pkv_pool* pool, int tokens, int in_features, int out_features, size_t* bytes)
{
    if (!pool || !bytes || tokens <= 0 || in_features <= 0 || out_features <= 0) return PKV_EINVAL;
    if (in_features % 64 || out_features % 128) return PKV_ENOTIMPL;
    if ((int64_t)tokens * out_features > ((int64_t)1 << 34) / 4) return PKV_ERANGE;
    *bytes = 0;  // split sums stay in the cluster's shared memory
    return PKV_OK;
}

int pkv_linear(pkv_pool* pool, const void* x, const void* w, void* y, int tokens, int in_features, int out_features,
               void* workspace, size_t workspace_bytes, void* stream)
{
    size_t need = 0;
    if (!pool || !x || !w || !y) return PKV_EINVAL;
    const int rc = pkv_linear_workspace_bytes(pool, tokens, in_features, out_features, &need);
    if (rc != PKV_OK) return rc;
    if (tokens > (1 << 24) || out_features > (1 << 20) || in_features > (1 << 20)) return PKV_ERANGE;
    if (!aligned(x, 16) || !aligned(w, 16) || !aligned(y, 16)) return PKV_EINVAL;
    if (need && (!workspace || workspace_bytes < need || !aligned(workspace, 256))) return PKV_EWORKSPACE;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != pool->device) return PKV_EDEVICE;
    void* ys[1] = {y};
    const int widths[1] = {out_features};
    return launch_linear(pool, x, w, tokens, in_features, 1, ys, widths, static_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? PKV_OK
               : PKV_ECUDA;
}

int pkv_qkv_proj(pkv_pool* pool, const void* x, const void* w_qkv, int tokens, int hidden, void* q, void* k, void* v,
                 void* stream)
{
    if (!pool || !x || !w_qkv || !q || !k || !v) return PKV_EINVAL;
    if (tokens <= 0 || hidden <= 0) return PKV_EINVAL;
    if (hidden % 64) return PKV_ENOTIMPL;
    if (tokens > (1 << 24) || hidden > (1 << 20)) return PKV_ERANGE;
    if (!aligned(x, 16) || !aligned(w_qkv, 16) || !aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16))
        return PKV_EINVAL;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != pool->device) return PKV_EDEVICE;
    const int qw = pool->cfg.heads * pool->cfg.head_dim, kw = pool->cfg.kv_heads * pool->cfg.head_dim;
    void* ys[3] = {q, k, v};
    const int widths[3] = {qw, kw, kw};
    return launch_linear(pool, x, w_qkv, tokens, hidden, 3, ys, widths, static_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? PKV_OK
               : PKV_ECUDA;
}

int pkv_output_gate(pkv_pool* pool, void* out, const void* gate, int tokens, void* stream)
{
    if (!pool || !out || !gate || tokens <= 0) return PKV_EINVAL;
    if (tokens > (1 << 24)) return PKV_ERANGE;
    if (!aligned(out, 16) || !aligned(gate, 16)) return PKV_EINVAL;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != pool->device) return PKV_EDEVICE;
    const int64_t n = (int64_t)tokens * pool->cfg.heads * pool->cfg.head_dim;
    return launch_gate(pool, out, gate, n, static_cast<cudaStream_t>(stream)) == cudaSuccess ? PKV_OK : PKV_ECUDA;
}

int pkv_check_errors(pkv_pool* pool, void* stream, uint32_t* flags)
{
    if (!pool || !flags) return PKV_EINVAL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return PKV_ECUDA;
    uint32_t h = 0;
    if (cudaMemcpy(&h, pool->err, sizeof h, cudaMemcpyDeviceToHost) != cudaSuccess) return PKV_ECUDA;
    if (cudaMemset(pool->err, 0, sizeof h) != cudaSuccess) return PKV_ECUDA;
    *flags = h;
    return PKV_OK;
}

int pkv_set_ctas(pkv_pool* pool, int ctas)
{
    if (!pool || ctas < 0) return PKV_EINVAL;
    pool->ctas_override = ctas;
    return PKV_OK;
}

int pkv_set_wait_limit(pkv_pool* pool, int64_t ns)
{
    if (!pool || ns < 0) return PKV_EINVAL;
    pool->wait_ns = (uint64_t)ns;
    return PKV_OK;
}

int pkv_timer_enable(pkv_pool* pool, int enable)
{
    if (!pool) return PKV_EINVAL;
    if (enable && !pool->ev_start) {
        pool->ev_start = new (std::nothrow) cudaEvent_t[kTimerSlots];
        pool->ev_stop = new (std::nothrow) cudaEvent_t[kTimerSlots];
        if (!pool->ev_start || !pool->ev_stop) return PKV_ENOMEM;
        for (int i = 0; i < kTimerSlots; ++i) {
            if (cudaEventCreate(&pool->ev_start[i]) != cudaSuccess ||
                cudaEventCreate(&pool->ev_stop[i]) != cudaSuccess)
                return PKV_ECUDA;
        }
    }
    if (enable < 0 || enable > 2) return PKV_EINVAL;
    pool->timer_on = enable;
    pool->timer_count = 0;
    return PKV_OK;
}

int pkv_timer_read(pkv_pool* pool, double* total_ms, int64_t* launches)
{
    if (!pool || !total_ms || !launches) return PKV_EINVAL;
    *total_ms = 0.0;
    *launches = 0;
    const int64_t cnt = pool->timer_count.load();
    if (!pool->ev_start || cnt == 0) return PKV_OK;
    const int64_t n = cnt < kTimerSlots ? cnt : kTimerSlots;
    const int last = (int)((cnt - 1) % kTimerSlots);
    if (cudaEventSynchronize(pool->ev_stop[last]) != cudaSuccess) return PKV_ECUDA;
    double sum = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        const int sl = (int)((cnt - 1 - i) % kTimerSlots);
        float ms = 0.f;
        if (cudaEventElapsedTime(&ms, pool->ev_start[sl], pool->ev_stop[sl]) != cudaSuccess) return PKV_ECUDA;
        sum += ms;
    }
    *total_ms = sum;
    *launches = n;
    return PKV_OK;
}

}  // extern "C"
