// race_api.cu -- the C ABI of librace_attn.so: argument checks, work planning, workspace
// carving and kernel dispatch.  Declarations and the contract of each entry point are in
// include/race_attn.h.
#include <cmath>
#include <mutex>
#include <string>
#include <type_traits>
#include <vector>

#include "race_attn.h"
#include "race_launch.h"

namespace race {

// ------------------------------------------------------------------ instrumentation

namespace {

struct ProfEntry {
    std::string name;
    int64_t launches = 0;
    double ms = 0.0;
    std::vector<std::pair<cudaEvent_t, cudaEvent_t>> pending;
};

uint64_t g_launches = 0;
bool g_profiling = false;
std::vector<ProfEntry> g_prof;
std::vector<cudaEvent_t> g_event_pool;
cudaEvent_t g_open_start = nullptr;

cudaEvent_t take_event()
{
    if (!g_event_pool.empty()) {
        cudaEvent_t e = g_event_pool.back();
        g_event_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

ProfEntry &entry(const char *name)
{
    for (auto &p : g_prof)
        if (p.name == name) return p;
    g_prof.push_back(ProfEntry{});
    g_prof.back().name = name;
    return g_prof.back();
}

void drain()
{
    for (auto &p : g_prof) {
        for (auto &ev : p.pending) {
            float ms = 0.f;
            if (cudaEventSynchronize(ev.second) == cudaSuccess &&
                cudaEventElapsedTime(&ms, ev.first, ev.second) == cudaSuccess) {
                p.ms += ms;
                p.launches += 1;
            }
            g_event_pool.push_back(ev.first);
            g_event_pool.push_back(ev.second);
        }
        p.pending.clear();
    }
}

}  // namespace

void prof_before(const char *, cudaStream_t st)
{
    ++g_launches;
    if (!g_profiling) return;
    g_open_start = take_event();
    if (g_open_start) cudaEventRecord(g_open_start, st);
}

void prof_after(const char *name, cudaStream_t st)
{
    if (!g_profiling || !g_open_start) return;
    cudaEvent_t e1 = take_event();
    if (!e1) return;
    cudaEventRecord(e1, st);
    entry(name).pending.emplace_back(g_open_start, e1);
    g_open_start = nullptr;
}

// ------------------------------------------------------------------ planning

namespace {
constexpr int kMaxDevices = 64;
int g_sm_count[kMaxDevices] = {};  // per device, filled on first use
}  // namespace

int device_sm_count()
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return 152;
    }
    int *cache = g_sm_count;
    if (cache[dev] > 0) return cache[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        n = 152;
    }
    cache[dev] = n;
    return n;
}

namespace {

constexpr size_t kMaxSmem = 227 * 1024;

int g_withhold = 0;  // failure-path test hook (race_attn_test_withhold_first_load)

struct Plan {
    Dims D{};
    bool causal = false, bf16 = false;
    bool nc5 = false;      // non-causal bf16 problem on the tcgen05 kernels
    bool c5 = false;       // causal bf16 problem whose forward runs on the tcgen05 kernels
    int nsplit = 1;        // token ranges (non-causal) or segments (causal) per (b, h)
    int64_t seg_len = 0;   // tokens per range, a multiple of the token tile
    size_t E = 0;          // floats per sketch: LR * (d + 1)
    size_t off_status = 0;  // one 32-bit device status word (error bits of bounded waits)
    size_t off_part = 0, off_sk = 0, off_gpart = 0, off_gsk = 0, off_aux = 0;
    size_t off_db = 0;     // d(loss)/d(beta) partials: [2][BH][db_cap] floats
    size_t off_fq = 0;     // causal tcgen05 backward: F'_Q rows handed from the query to the key side
    size_t off_fk = 0;     // causal tcgen05 path without `state`: the keys' bucket-feature rows,
    size_t off_kinv = 0;   //   then their 1 / |k|
    size_t state_fk = 0;   // causal tcgen05 path: the same two arrays inside `state`
    size_t state_kinv = 0;
    int64_t db_cap = 0;    // partial slots per (side, b, h): at least every backward kernel's grid x
    size_t off_dzq = 0, off_dzk = 0, off_dwpart = 0;  // d(loss)/d(W): dz / |x| rows, then partials
    int dw_nblk = 1;       // token ranges per (b, h) of the d(loss)/d(W) reduction
    size_t ws_fwd = 0, ws_bwd = 0, ws_bwd_dw = 0, state = 0;
};

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

int make_plan(const race_shape *s, int L, int P, int causal, Plan &pl)
{
    if (!s) return RACE_ERR_INVALID_ARG;
    if (s->B < 1 || s->H < 1 || s->N < 1) return RACE_ERR_INVALID_ARG;  // B * H <= 65535 below
    if (s->d < 8 || s->d > kMaxD || s->d % 8 != 0) return RACE_ERR_INVALID_ARG;
    if (P < 1 || P > kMaxP || L < 1 || L > kMaxL) return RACE_ERR_INVALID_ARG;
    if ((L << P) > kMaxLR) return RACE_ERR_INVALID_ARG;
    if (s->dtype != RACE_F32 && s->dtype != RACE_BF16) return RACE_ERR_INVALID_ARG;
    if (s->per_head_w != 0 && s->per_head_w != 1) return RACE_ERR_INVALID_ARG;
    if (s->B > 65535 || s->H > 65535 || s->B * s->H > 65535 || s->N > ((int64_t)1 << 40) / (s->B * s->H))
        return RACE_ERR_INVALID_ARG;
    Dims &D = pl.D;
    D.BH = s->B * s->H;
    D.N = s->N;
    D.d = (int)s->d;
    D.L = L;
    D.P = P;
    D.R = 1 << P;
    D.LR = L << P;
    D.LP = L * P;
    D.dv = D.d + 1;
    D.beta = 0.f;
    D.H = s->H;
    D.w_per_head = s->per_head_w;
    D.sms = device_sm_count();
    D.withhold = 0;
    pl.causal = causal != 0;
    pl.bf16 = s->dtype == RACE_BF16;
    pl.E = (size_t)D.LR * D.dv;

    pl.nc5 = !pl.causal && pl.bf16 && nc5_supported(D);
    pl.c5 = pl.causal && pl.bf16 && c5_supported(D);
    // segment granule: a multiple of every kernel's token tile
    const int TT = (pl.nc5 || pl.c5) ? nc5_tile() : 64;
    const int64_t ntiles = ceil_div(D.N, TT);
    int64_t want;
    if (pl.nc5) {
        want = ceil_div((int64_t)D.sms * nc5_sketch_ctas_per_sm(D), D.BH);
    } else if (!pl.causal) {
        const int64_t chunks = ceil_div(D.LR, 64);
        want = ceil_div(4 * (int64_t)D.sms, chunks * D.BH);
    } else {
        want = ceil_div(2 * (int64_t)D.sms, D.BH);
    }
    want = std::max<int64_t>(1, std::min(want, ntiles));
    pl.seg_len = ceil_div(ceil_div(D.N, want), TT) * TT;
    pl.nsplit = (int)ceil_div(D.N, pl.seg_len);

    const size_t sk_one = pl.E * sizeof(float);
    const size_t per_split = (size_t)D.BH * pl.nsplit * sk_one;
    const size_t per_bh = (size_t)D.BH * sk_one;
    pl.off_status = 0;
    pl.off_part = 256;
    pl.off_sk = align256(pl.off_part + per_split);
    const size_t sk_bytes = pl.causal ? per_split : per_bh;
    // the causal tcgen05 path keeps every key's bucket features (bf16) from the segment-sum pass
    const size_t fk_bytes = pl.c5 ? c5_feature_rows_bytes(D) : 0;
    const size_t kinv_bytes = pl.c5 ? (size_t)D.BH * D.N * sizeof(float) : 0;
    pl.off_fk = align256(pl.off_sk + sk_bytes);
    pl.off_kinv = align256(pl.off_fk + fk_bytes);
    pl.ws_fwd = align256(pl.off_kinv + kinv_bytes);
    pl.off_gpart = pl.ws_fwd;
    pl.off_gsk = align256(pl.off_gpart + per_split);
    pl.off_aux = align256(pl.off_gsk + sk_bytes);
    pl.off_db = align256(pl.off_aux + (size_t)D.BH * D.N * sizeof(float2));
    pl.db_cap = std::max<int64_t>(pl.nsplit, ceil_div(D.N, generic_token_tile()));
    pl.off_fq = align256(pl.off_db + 2 * (size_t)D.BH * pl.db_cap * sizeof(float));
    const size_t fq_bytes = (pl.c5 && c5_bwd_supported(D)) ? c5_feature_rows_bytes(D) : 0;
    pl.ws_bwd = align256(pl.off_fq + fq_bytes);
    pl.dw_nblk = (int)std::max<int64_t>(1, std::min(ceil_div(D.N, 32), ceil_div(4 * (int64_t)D.sms, D.BH)));
    D.dzld = (D.LP + 3) & ~3;
    const size_t dz_bytes = (size_t)D.BH * D.N * D.dzld * sizeof(float);
    pl.off_dzq = pl.ws_bwd;
    pl.off_dzk = align256(pl.off_dzq + dz_bytes);
    pl.off_dwpart = align256(pl.off_dzk + dz_bytes);
    pl.ws_bwd_dw = align256(pl.off_dwpart + (size_t)D.BH * pl.dw_nblk * D.LP * D.d * sizeof(float));
    pl.state_fk = align256(sk_bytes);
    pl.state_kinv = align256(pl.state_fk + fk_bytes);
    pl.state = pl.c5 ? pl.state_kinv + kinv_bytes : sk_bytes;

    // every kernel of the chosen path must fit in shared memory
    if (pl.causal) {
        if (generic_smem_bytes(D, GenericKernel::CausalBwd) > kMaxSmem ||
            generic_smem_bytes(D, GenericKernel::CausalFwd) > kMaxSmem)
            return RACE_ERR_UNSUPPORTED;
    } else {
        if (generic_smem_bytes(D, GenericKernel::QueryBwd) > kMaxSmem ||
            generic_smem_bytes(D, GenericKernel::KeyBwd) > kMaxSmem ||
            generic_smem_bytes(D, GenericKernel::Readout) > kMaxSmem)
            return RACE_ERR_UNSUPPORTED;
    }
    if (generic_smem_bytes(D, GenericKernel::Sketch) > kMaxSmem) return RACE_ERR_UNSUPPORTED;
    return RACE_OK;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15) == 0; }

// The status a device status word reports: a timed-out wait first (its outputs are incomplete),
// then a degenerate denominator.
int status_of(unsigned bits)
{
    if (bits & kErrTimeout) return RACE_ERR_DEVICE_TIMEOUT;
    if (bits & kErrNumeric) return RACE_ERR_NUMERIC;
    return RACE_OK;
}

// beta: finite and >= 0, or +infinity for hard hashing.
int check_beta(float beta) { return (!std::isnan(beta) && beta >= 0.f) ? RACE_OK : RACE_ERR_INVALID_ARG; }

// Hard hashing (beta = +infinity, the limit "RACE Attention" slides, frame "Soft corner assignments
// make hashing differentiable", call hard hashing) runs the soft kernels at the finite stand-in
// 2^126.  Their sigmoid(2 beta u) is then exactly 1 or 0 for every |u| >= 2^-119 (the exponent
// underflows) and exactly 1/2 at u = 0, the value a tied projection keeps in the limit.  So
// the features are the hard corners, and the softmax gradient vanishes identically.  Only tied
// rows (u = 0) would carry a Jacobian scaled by 2^126, and their dQ and dK are zero by definition.
constexpr float kHardBeta = 8.507059e37f;  // 2^126
bool hard_hash(float beta) { return std::isinf(beta); }
float kernel_beta(float beta) { return hard_hash(beta) ? kHardBeta : beta; }

#define RACE_TRY(expr)                                   \
    do {                                                 \
        cudaError_t e_ = (expr);                         \
        if (e_ != cudaSuccess) return RACE_ERR_CUDA;     \
    } while (0)

template <typename T>
int forward_impl(const Plan &pl, const T *Q, const T *K, const T *V, const float *W, T *O, float *state,
                 char *ws, cudaStream_t st)
{
    const Dims &D = pl.D;
    float *part = (float *)(ws + pl.off_part);
    float *S = state ? state : (float *)(ws + pl.off_sk);
    unsigned *err = (unsigned *)(ws + pl.off_status);
    RACE_TRY(cudaMemsetAsync(err, 0, sizeof(unsigned), st));
    if constexpr (std::is_same<T, bf16_t>::value) {
        if (pl.c5) {
            // segment sums of the causal sketch = the non-causal sketch of each segment; the pass
            // also stores every key's bucket features, which the chunk kernel reads instead of K
            bf16_t *fk = state ? (bf16_t *)((char *)state + pl.state_fk) : (bf16_t *)(ws + pl.off_fk);
            float *kinv = state ? (float *)((char *)state + pl.state_kinv) : (float *)(ws + pl.off_kinv);
            RACE_TRY(launch_nc5_sketch(D, K, V, nullptr, W, pl.seg_len, pl.nsplit, part, err, st, fk, kinv));
            RACE_TRY(launch_combine(D, part, S, pl.nsplit, 1, st));
            RACE_TRY(launch_c5_fwd(D, Q, fk, V, W, S, pl.seg_len, pl.nsplit, O, err, st));
            return RACE_OK;
        }
    }
    if constexpr (std::is_same<T, bf16_t>::value) {
        if (pl.nc5) {
            RACE_TRY(launch_nc5_sketch(D, K, V, nullptr, W, pl.seg_len, pl.nsplit, part, err, st));
            RACE_TRY(launch_combine(D, part, S, pl.nsplit, 0, st));
            RACE_TRY(launch_nc5_readout(D, Q, W, S, O, err, st));
            return RACE_OK;
        }
    }
    RACE_TRY(launch_sketch<T>(D, K, V, nullptr, W, pl.seg_len, pl.nsplit, part, 0, st));
    if (!pl.causal) {
        RACE_TRY(launch_combine(D, part, S, pl.nsplit, 0, st));
        RACE_TRY(launch_readout<T>(D, Q, W, S, O, err, st));
    } else {
        RACE_TRY(launch_combine(D, part, S, pl.nsplit, 1, st));
        RACE_TRY(launch_causal_fwd<T>(D, Q, K, V, W, S, pl.seg_len, pl.nsplit, O, err, st));
    }
    return RACE_OK;
}

// d(loss)/d(beta): each backward kernel's CTA (slot x, b, h) writes one partial of its side to
// dbq / dbk[(b, h) * slots + x]; a fixed-order combine then sums both sides into dbeta[b, h].
struct DbetaOut {
    float *dbq = nullptr, *dbk = nullptr, *out = nullptr;
    int slots = 0;
};

cudaError_t dbeta_begin(const Plan &pl, char *ws, float *dbeta, int slots, DbetaOut &db, cudaStream_t st)
{
    // the kernels' d(beta) instances also write the rows' dz when d(loss)/d(W) is asked for, so
    // they run then too (their d(beta) partials go unused without a dbeta output)
    if (!dbeta && pl.D.dzq == nullptr) return cudaSuccess;
    db.slots = slots;
    db.out = dbeta;
    db.dbq = (float *)(ws + pl.off_db);
    db.dbk = db.dbq + pl.D.BH * slots;
    return cudaMemsetAsync(db.dbq, 0, 2 * (size_t)pl.D.BH * slots * sizeof(float), st);
}

cudaError_t dbeta_end(const Plan &pl, const DbetaOut &db, cudaStream_t st)
{
    if (!db.out) return cudaSuccess;
    return launch_dbeta_combine(pl.D, db.dbq, db.slots, db.out, st);
}

template <typename T>
int backward_impl(const Plan &pl, const T *Q, const T *K, const T *V, const float *W, const T *dO, T *dQ, T *dK,
                  T *dV, float *dbeta, const float *state, char *ws, cudaStream_t st)
{
    const Dims &D = pl.D;
    float *part = (float *)(ws + pl.off_part);
    float *gpart = (float *)(ws + pl.off_gpart);
    float *gsk = (float *)(ws + pl.off_gsk);
    float2 *aux = (float2 *)(ws + pl.off_aux);
    unsigned *err = (unsigned *)(ws + pl.off_status);
    RACE_TRY(cudaMemsetAsync(err, 0, sizeof(unsigned), st));
    const float *S = state;
    DbetaOut db;
    if constexpr (std::is_same<T, bf16_t>::value) {
        if (pl.c5 && c5_bwd_supported(D)) {
            // the keys' bucket-feature rows: from the forward's state, or stored again here
            const bf16_t *fk = S ? (const bf16_t *)((const char *)S + pl.state_fk) : (const bf16_t *)(ws + pl.off_fk);
            const float *kinv = S ? (const float *)((const char *)S + pl.state_kinv) : (const float *)(ws + pl.off_kinv);
            if (!S) {
                float *Sw = (float *)(ws + pl.off_sk);
                RACE_TRY(launch_nc5_sketch(D, K, V, nullptr, W, pl.seg_len, pl.nsplit, part, err, st,
                                           (bf16_t *)(ws + pl.off_fk), (float *)(ws + pl.off_kinv)));
                RACE_TRY(launch_combine(D, part, Sw, pl.nsplit, 1, st));
                S = Sw;
            }
            RACE_TRY(dbeta_begin(pl, ws, dbeta, pl.nsplit, db, st));
            bf16_t *fq = (bf16_t *)(ws + pl.off_fq);
            RACE_TRY(launch_c5_bwd_q(D, Q, fk, V, dO, W, S, pl.seg_len, pl.nsplit, dQ, aux, fq, gpart, err, db.dbq,
                                     st));
            RACE_TRY(launch_combine(D, gpart, gsk, pl.nsplit, 2, st));
            RACE_TRY(launch_c5_bwd_kv(D, fq, fk, kinv, K, V, dO, aux, W, gsk, pl.seg_len, pl.nsplit, dK, dV, err,
                                      db.dbk, st));
            RACE_TRY(dbeta_end(pl, db, st));
            return RACE_OK;
        }
    }
    if constexpr (std::is_same<T, bf16_t>::value) {
        if (pl.nc5) {
            if (!S) {
                float *Sw = (float *)(ws + pl.off_sk);
                RACE_TRY(launch_nc5_sketch(D, K, V, nullptr, W, pl.seg_len, pl.nsplit, part, err, st));
                RACE_TRY(launch_combine(D, part, Sw, pl.nsplit, 0, st));
                S = Sw;
            }
            RACE_TRY(dbeta_begin(pl, ws, dbeta, nc5_bwd_nseg(D), db, st));
            RACE_TRY(launch_nc5_bwd_query(D, Q, dO, W, S, dQ, aux, err, db.dbq, st));
            RACE_TRY(launch_nc5_sketch(D, Q, dO, aux, W, pl.seg_len, pl.nsplit, gpart, err, st));
            RACE_TRY(launch_combine(D, gpart, gsk, pl.nsplit, 0, st));
            RACE_TRY(launch_nc5_bwd_key(D, K, V, W, gsk, dK, dV, err, db.dbk, st));
            RACE_TRY(dbeta_end(pl, db, st));
            return RACE_OK;
        }
    }
    if (!S) {
        float *Sw = (float *)(ws + pl.off_sk);
        RACE_TRY(launch_sketch<T>(D, K, V, nullptr, W, pl.seg_len, pl.nsplit, part, 0, st));
        RACE_TRY(launch_combine(D, part, Sw, pl.nsplit, pl.causal ? 1 : 0, st));
        S = Sw;
    }
    if (!pl.causal) {
        RACE_TRY(dbeta_begin(pl, ws, dbeta, (int)ceil_div(D.N, generic_token_tile()), db, st));
        RACE_TRY(launch_bwd_query<T>(D, Q, dO, W, S, dQ, aux, db.dbq, st));
        RACE_TRY(launch_sketch<T>(D, Q, dO, aux, W, pl.seg_len, pl.nsplit, gpart, 1, st));
        RACE_TRY(launch_combine(D, gpart, gsk, pl.nsplit, 0, st));
        RACE_TRY(launch_bwd_key<T>(D, K, V, W, gsk, dK, dV, db.dbk, st));
    } else {
        RACE_TRY(dbeta_begin(pl, ws, dbeta, pl.nsplit, db, st));
        RACE_TRY(launch_causal_bwd_q<T>(D, Q, K, V, dO, W, S, pl.seg_len, pl.nsplit, dQ, aux, db.dbq, st));
        RACE_TRY(launch_sketch<T>(D, Q, dO, aux, W, pl.seg_len, pl.nsplit, gpart, 1, st));
        RACE_TRY(launch_combine(D, gpart, gsk, pl.nsplit, 2, st));
        RACE_TRY(launch_causal_bwd_kv<T>(D, Q, K, V, dO, aux, W, gsk, pl.seg_len, pl.nsplit, dK, dV, db.dbk, st));
    }
    RACE_TRY(dbeta_end(pl, db, st));
    return RACE_OK;
}

}  // namespace
}  // namespace race

using namespace race;

extern "C" {

size_t race_attn_workspace_bytes(const race_shape *shape, int L, int P, int causal, int is_bwd)
{
    Plan pl;
    if (make_plan(shape, L, P, causal, pl) != RACE_OK) return 0;
    return is_bwd == 2 ? pl.ws_bwd_dw : is_bwd ? pl.ws_bwd : pl.ws_fwd;
}

size_t race_attn_state_bytes(const race_shape *shape, int L, int P, int causal)
{
    Plan pl;
    if (make_plan(shape, L, P, causal, pl) != RACE_OK) return 0;
    return pl.state;
}

int race_attn_fwd(const race_shape *shape, const void *Q, const void *K, const void *V, const float *W, float beta,
                  int L, int P, int causal, void *O, void *state, void *workspace, size_t workspace_bytes,
                  void *stream)
{
    Plan pl;
    int rc = make_plan(shape, L, P, causal, pl);
    if (rc != RACE_OK) return rc;
    if ((rc = check_beta(beta)) != RACE_OK) return rc;
    if (!Q || !K || !V || !W || !O || !workspace) return RACE_ERR_INVALID_ARG;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(W) || !aligned16(O) ||
        !aligned16(workspace) || (state && !aligned16(state)))
        return RACE_ERR_ALIGN;
    if (workspace_bytes < pl.ws_fwd) return RACE_ERR_WORKSPACE;
    pl.D.beta = kernel_beta(beta);
    pl.D.withhold = g_withhold;
    cudaStream_t st = (cudaStream_t)stream;
    if (pl.bf16)
        return forward_impl<__nv_bfloat16>(pl, (const __nv_bfloat16 *)Q, (const __nv_bfloat16 *)K,
                                           (const __nv_bfloat16 *)V, W, (__nv_bfloat16 *)O, (float *)state,
                                           (char *)workspace, st);
    return forward_impl<float>(pl, (const float *)Q, (const float *)K, (const float *)V, W, (float *)O,
                               (float *)state, (char *)workspace, st);
}

int race_attn_bwd(const race_shape *shape, const void *Q, const void *K, const void *V, const float *W, float beta,
                  int L, int P, int causal, const void *O, const void *dO, void *dQ, void *dK, void *dV,
                  float *dbeta, float *dW, const void *state, void *workspace, size_t workspace_bytes,
                  void *stream)
{
    (void)O;
    Plan pl;
    int rc = make_plan(shape, L, P, causal, pl);
    if (rc != RACE_OK) return rc;
    if ((rc = check_beta(beta)) != RACE_OK) return rc;
    if (!Q || !K || !V || !W || !dO || !dQ || !dK || !dV || !workspace) return RACE_ERR_INVALID_ARG;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(W) || !aligned16(dO) || !aligned16(dQ) ||
        !aligned16(dK) || !aligned16(dV) || !aligned16(workspace) || (state && !aligned16(state)) ||
        ((uintptr_t)dbeta & 3) != 0 || ((uintptr_t)dW & 3) != 0)
        return RACE_ERR_ALIGN;
    if (workspace_bytes < (dW ? pl.ws_bwd_dw : pl.ws_bwd)) return RACE_ERR_WORKSPACE;
    pl.D.beta = kernel_beta(beta);
    cudaStream_t st = (cudaStream_t)stream;
    const bool want_dw = dW != nullptr && !hard_hash(beta);
    if (want_dw) {  // the backward kernels also write every row's dz / |x|
        pl.D.dzq = (float *)((char *)workspace + pl.off_dzq);
        pl.D.dzk = (float *)((char *)workspace + pl.off_dzk);
        if (pl.D.LP & 3)  // the rows' padding past L P, which not every kernel family writes, reads as 0
            RACE_TRY(cudaMemsetAsync(pl.D.dzq, 0, pl.off_dwpart - pl.off_dzq, st));
    }
    if (pl.bf16)
        rc = backward_impl<__nv_bfloat16>(pl, (const __nv_bfloat16 *)Q, (const __nv_bfloat16 *)K,
                                          (const __nv_bfloat16 *)V, W, (const __nv_bfloat16 *)dO,
                                          (__nv_bfloat16 *)dQ, (__nv_bfloat16 *)dK, (__nv_bfloat16 *)dV, dbeta,
                                          (const float *)state, (char *)workspace, st);
    else
        rc = backward_impl<float>(pl, (const float *)Q, (const float *)K, (const float *)V, W, (const float *)dO,
                                  (float *)dQ, (float *)dK, (float *)dV, dbeta, (const float *)state,
                                  (char *)workspace, st);
    if (rc == RACE_OK && want_dw) {
        float *dwpart = (float *)((char *)workspace + pl.off_dwpart);
        if (pl.bf16)
            RACE_TRY(launch_dw(pl.D, (const __nv_bfloat16 *)Q, (const __nv_bfloat16 *)K, pl.dw_nblk, dwpart, dW, st));
        else
            RACE_TRY(launch_dw(pl.D, (const float *)Q, (const float *)K, pl.dw_nblk, dwpart, dW, st));
    }
    if (rc == RACE_OK && hard_hash(beta)) {  // a hard hash passes no gradient to Q, K or W
        const size_t bytes = (size_t)pl.D.BH * pl.D.N * pl.D.d * (pl.bf16 ? 2 : 4);
        RACE_TRY(cudaMemsetAsync(dQ, 0, bytes, st));
        RACE_TRY(cudaMemsetAsync(dK, 0, bytes, st));
        if (dW) RACE_TRY(cudaMemsetAsync(dW, 0, (size_t)pl.D.BH * pl.D.LP * pl.D.d * sizeof(float), st));
    }
    return rc;
}

const char *race_attn_strerror(int status)
{
    switch (status) {
        case RACE_OK: return "ok";
        case RACE_ERR_INVALID_ARG: return "invalid argument";
        case RACE_ERR_UNSUPPORTED: return "unsupported problem size for this build";
        case RACE_ERR_WORKSPACE: return "workspace too small";
        case RACE_ERR_CUDA: return "CUDA launch or runtime error";
        case RACE_ERR_ALIGN: return "tensor pointer not 16-byte aligned";
        case RACE_ERR_SCRATCH_LIMIT: return "problem needs more scratch than the built-in no-alloc buffer";
        case RACE_ERR_DEVICE_TIMEOUT: return "a kernel gave up waiting for an asynchronous copy";
        case RACE_ERR_NUMERIC: return "an output row has a zero, negative or non-finite denominator";
        case RACE_ERR_NOALLOC_SETUP:
            return "the built-in no-alloc scratch could not be set up on this device (out of memory, or first use "
                   "inside a stream capture: call race_attn_noalloc_init first)";
        default: return "unknown status";
    }
}

int race_attn_decode(const race_shape *shape, const void *q, const void *k, const void *v, const float *W,
                     float beta, int L, int P, void *state, void *o, void *stream)
{
    Plan pl;
    int rc = make_plan(shape, L, P, 0, pl);
    if (rc != RACE_OK) return rc;
    if (shape->N != 1 || check_beta(beta) != RACE_OK) return RACE_ERR_INVALID_ARG;
    if (!q || !k || !v || !W || !state || !o) return RACE_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(W) || !aligned16(state) || !aligned16(o))
        return RACE_ERR_ALIGN;
    if (!decode_supported(pl.D)) return RACE_ERR_UNSUPPORTED;
    Dims D = pl.D;
    D.beta = kernel_beta(beta);
    cudaStream_t st = (cudaStream_t)stream;
    if (pl.bf16)
        RACE_TRY(launch_decode<bf16_t>(D, (const bf16_t *)q, (const bf16_t *)k, (const bf16_t *)v, W, (float *)state,
                                       (bf16_t *)o, st));
    else
        RACE_TRY(launch_decode<float>(D, (const float *)q, (const float *)k, (const float *)v, W, (float *)state,
                                      (float *)o, st));
    return RACE_OK;
}

int race_attn_angular(const race_shape *shape, const void *Q, const void *K, const void *V, float gamma, int causal,
                      void *O, void *stream)
{
    Plan pl;
    int rc = make_plan(shape, 1, 1, causal, pl);  // shape checks only: this path has no tables
    if (rc != RACE_OK) return rc;
    if (!std::isfinite(gamma) || gamma < 0.f) return RACE_ERR_INVALID_ARG;
    if (!Q || !K || !V || !O) return RACE_ERR_INVALID_ARG;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O)) return RACE_ERR_ALIGN;
    cudaStream_t st = (cudaStream_t)stream;
    if (pl.bf16)
        RACE_TRY(launch_angular<bf16_t>(pl.D, (const bf16_t *)Q, (const bf16_t *)K, (const bf16_t *)V, gamma,
                                        causal != 0, (bf16_t *)O, st));
    else
        RACE_TRY(launch_angular<float>(pl.D, (const float *)Q, (const float *)K, (const float *)V, gamma,
                                       causal != 0, (float *)O, st));
    return RACE_OK;
}

int race_attn_status(const void *workspace, void *stream)
{
    if (!workspace) return RACE_ERR_INVALID_ARG;
    unsigned bits = 0;
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return RACE_ERR_CUDA;
    if (cudaMemcpy(&bits, workspace, sizeof bits, cudaMemcpyDeviceToHost) != cudaSuccess) return RACE_ERR_CUDA;
    return status_of(bits);
}

int race_attn_test_withhold_first_load(int enable)
{
    g_withhold = enable != 0;
    return RACE_OK;
}

uint64_t race_attn_launch_count(void) { return g_launches; }

int race_attn_profile(int enable)
{
    g_profiling = enable != 0;
    return RACE_OK;
}

int race_attn_profile_read(int i, const char **name, int64_t *launches, double *total_ms)
{
    drain();
    const int n = (int)g_prof.size();
    if (i < 0 || i >= n) return i == 0 && n == 0 ? 0 : -1;
    if (name) *name = g_prof[i].name.c_str();
    if (launches) *launches = g_prof[i].launches;
    if (total_ms) *total_ms = g_prof[i].ms;
    return n;
}

void race_attn_profile_reset(void)
{
    drain();
    g_prof.clear();
}

}  // extern "C"

// ------------------------------------------------------------------ forward without a workspace
//
// Scratch for race_attn_fwd_noalloc: a static device array, so callers that may not allocate
// device memory can still run the forward pass.  Host code must not use the symbol itself as a
// pointer (on the host it names a shadow variable, not device memory); the device address is
// looked up once per device with cudaGetSymbolAddress and cached.

namespace race {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[RACE_NOALLOC_SCRATCH_BYTES];
std::mutex g_noalloc_mutex;
void *g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up on first use (which,
// under lazy module loading, is when the driver loads the array).  `st`: the caller's stream,
// checked for an ongoing capture before a first use when check_capture is set.
int noalloc_scratch(cudaStream_t st, bool check_capture, void **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return RACE_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_ptr[dev]) {
        if (check_capture) {
            cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
            if (cudaStreamIsCapturing(st, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) {
                cudaGetLastError();
                return RACE_ERR_NOALLOC_SETUP;
            }
        }
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return e == cudaErrorMemoryAllocation ? RACE_ERR_NOALLOC_SETUP : RACE_ERR_CUDA;
        }
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return RACE_OK;
}

}  // namespace
}  // namespace race

extern "C" int race_attn_noalloc_init(void)
{
    void *p = nullptr;
    return noalloc_scratch(nullptr, false, &p);
}

extern "C" int race_attn_noalloc_status(void *stream)
{
    void *p = nullptr;
    {
        int dev = -1;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return RACE_ERR_CUDA;
        std::lock_guard<std::mutex> lock(g_noalloc_mutex);
        p = g_noalloc_ptr[dev];
    }
    if (!p) return RACE_OK;  // no allocation-free call has run on this device
    return race_attn_status(p, stream);
}

extern "C" int race_attn_fwd_noalloc(const race_shape *shape, const void *Q, const void *K, const void *V,
                                     const float *W, float beta, int L, int P, int causal, void *O, void *stream)
{
    Plan pl;
    int rc = make_plan(shape, L, P, causal, pl);
    if (rc != RACE_OK) return rc;
    if ((rc = check_beta(beta)) != RACE_OK) return rc;
    if (!Q || !K || !V || !W || !O) return RACE_ERR_INVALID_ARG;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(W) || !aligned16(O)) return RACE_ERR_ALIGN;
    if (pl.ws_fwd > RACE_NOALLOC_SCRATCH_BYTES) return RACE_ERR_SCRATCH_LIMIT;
    cudaStream_t st = (cudaStream_t)stream;
    void *scratch = nullptr;
    if ((rc = noalloc_scratch(st, true, &scratch)) != RACE_OK) return rc;
    pl.D.beta = kernel_beta(beta);
    pl.D.withhold = g_withhold;
    // state == nullptr: the forward keeps its sketch inside the scratch buffer
    if (pl.bf16)
        return forward_impl<__nv_bfloat16>(pl, (const __nv_bfloat16 *)Q, (const __nv_bfloat16 *)K,
                                           (const __nv_bfloat16 *)V, W, (__nv_bfloat16 *)O, nullptr, (char *)scratch,
                                           st);
    return forward_impl<float>(pl, (const float *)Q, (const float *)K, (const float *)V, W, (float *)O, nullptr,
                               (char *)scratch, st);
}
