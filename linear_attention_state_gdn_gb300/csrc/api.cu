// api.cu -- the C ABI of libhypic (include/hypic.h): argument validation on the host,
// launch-table construction (segments in longest-first order) and kernel dispatch.
//
// Nothing here allocates device memory. The only device state the library keeps is one
// 4-byte status word per device (a file-scope __device__ variable), which kernels set
// when a bounded wait runs out or a gate leaves the supported range.
#include <algorithm>
#include <cstring>
#include <mutex>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "internal.cuh"
#include "ptx.cuh"

using namespace hypic;

namespace {

__device__ unsigned g_status_word;

constexpr int kMaxDevices = 64;
unsigned *g_status_addr[kMaxDevices];
std::mutex g_status_mu;

// Device address of this device's status word. Host code may not use &g_status_word
// (it names the host-side shadow), so the address is looked up once per device with
// that device current.
unsigned *status_word(int *dev_out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    if (dev_out) *dev_out = dev;
    std::lock_guard<std::mutex> lock(g_status_mu);
    if (!g_status_addr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_status_word) != cudaSuccess) return nullptr;
        g_status_addr[dev] = static_cast<unsigned *>(ptr);
    }
    return g_status_addr[dev];
}

// Library-owned build scratch for hypic_build_segments_static_ws: a file-scope device array
// (reserved when the module loads; nothing is allocated at call time), located once per
// device like the status word. No part of it needs to start at zero: the build overwrites
// every record it later reads.
__device__ __align__(256) unsigned char g_static_ws[HYPIC_STATIC_WS_BYTES];
void *g_static_ws_addr[kMaxDevices];

void *static_workspace() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_status_mu);
    if (!g_static_ws_addr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_static_ws) != cudaSuccess) return nullptr;
        g_static_ws_addr[dev] = ptr;
    }
    return g_static_ws_addr[dev];
}

// hypic_probe_wait_timeout: one warp per CTA allocates tensor memory as the kernels do; its
// first thread waits with the bounded wait on a barrier nothing arrives at (the limit runs
// out and sets kErrTimeout), raises the CTA's abort flag as a multi-role kernel's timed-out
// role does, and checks that a second wait gives up on that flag at once instead of sitting
// out its own limit; the warp then frees the tensor memory.
__global__ void __launch_bounds__(32) wait_probe_kernel(unsigned *err, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    __shared__ uint32_t tslot;
    __shared__ volatile int abort_flag;
    if (threadIdx.x == 0) {
        ptx::mbar_init(&bar, 1);
        abort_flag = 0;
        ptx::fence_mbar_init();
    }
    ptx::tmem_alloc(&tslot, 32);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = tslot;
    if (threadIdx.x == 0 && !ptx::mbar_wait(&bar, 0, err, kErrTimeout, limit_ns)) {
        abort_flag = 1;
        ptx::mbar_wait_or_abort(&bar, 0, err, kErrTimeout, &abort_flag);
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 32);
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// True if p is memory the current device can read with plain loads (device or managed).
bool on_device(const void *p) {
    if (!p) return false;
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    int dev = -1;
    cudaGetDevice(&dev);
    if (at.type == cudaMemoryTypeManaged) return true;
    return at.type == cudaMemoryTypeDevice && at.device == dev;
}

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    if (!a || !b || na == 0 || nb == 0) return false;
    const char *pa = static_cast<const char *>(a), *pb = static_cast<const char *>(b);
    return pa < pb + nb && pb < pa + na;
}

bool head_size_ok(int d_k, int d_v) {
    return d_k == d_v && (d_k == 32 || d_k == 64 || d_k == 128);
}

hypic_status from_cuda(cudaError_t e) { return e == cudaSuccess ? HYPIC_OK : HYPIC_ERR_CUDA; }

// A named NVTX range around an entry point: the call's launches show under its name in a
// profiler's timeline; without a profiler attached the push and pop return at once.
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};

enum class BuildPath { None, GatedSimt, GatedTc, Seq, GdnTc };

bool dense_family(int fam) { return fam == HYPIC_FAM_DELTA || fam == HYPIC_FAM_GDN || fam == HYPIC_FAM_KDA; }
enum class ComposePath { None, Scaled, DenseSimt, DenseTc, DenseCols };

// Kernel selection for a build (shape/family/dtype only; no pointer checks).
BuildPath pick_build(const hypic_build_args *a) {
    if (a->n_seg == 0) return BuildPath::None;
    // start states: the exact path; the segment outputs too, except on the tensor-core
    // DeltaNet / GDN build, whose outputs instance computes them
    if (a->S_init) return BuildPath::Seq;
    const bool delta = dense_family(a->family);
    if (a->O && (!delta || a->family == HYPIC_FAM_KDA)) return BuildPath::Seq;
    BuildParams q{};
    q.family = a->family;
    q.dtype = a->dtype;
    q.D = a->d_k;
    // the KDA preparation reads the per-channel log-gates of a channel pair as one 8-byte word
    if (a->family == HYPIC_FAM_KDA && (reinterpret_cast<uintptr_t>(a->log_gate) & 7u)) return BuildPath::Seq;
    if (delta) return build_gdn_tc_supported(q) ? BuildPath::GdnTc : BuildPath::Seq;
    return build_gated_tc_supported(q) ? BuildPath::GatedTc : BuildPath::GatedSimt;
}

ComposePath pick_compose(const hypic_compose_args *a) {
    if (a->n_seg == 0 || a->n_units == 0) return ComposePath::None;
    const bool dense = dense_family(a->family);
    if (!dense) return ComposePath::Scaled;
    ComposeParams q{};
    q.D = a->d_k;
    q.n_seg = a->n_seg;
    q.n_units = a->n_units;
    q.lam_total = a->lam_total;
    q.P_total = a->P_total;
    // a plain scan of few units: four CTAs per unit, each carrying a block of state columns
    if (compose_dense_cols_supported(q)) return ComposePath::DenseCols;
    return compose_dense_tc_supported(q) ? ComposePath::DenseTc : ComposePath::DenseSimt;
}

// Workspace records of the GDN / DeltaNet / KDA tensor-core build: one per (segment, value
// head, 64-token chunk). Negative segment lengths count as empty (they are rejected elsewhere).
int64_t gdn_records(const hypic_build_args *a) {
    int64_t records = 0;
    for (int j = 0; j < a->n_seg; ++j) {
        const int64_t len = a->seg_offsets[j + 1] - a->seg_offsets[j];
        if (len > 0) records += (int64_t)a->H_v * ((len + kGdnChunk - 1) / kGdnChunk);
    }
    return records;
}

// Bytes of the records: M2 per record, the tail (ticket counter), and for KDA the gated keys
// and log-decays (kKdaExtraBytes per record) after the tail.
size_t gdn_records_bytes(const hypic_build_args *a) {
    const size_t r = (size_t)gdn_records(a);
    return r * (size_t)kGdnRecordBytes + (size_t)kGdnWorkspaceTail +
           (a->family == HYPIC_FAM_KDA ? r * (size_t)kKdaExtraBytes : 0);
}

// Intra-segment split of the tensor-core builds (DeltaNet / GDN, and the linear / scalar /
// diagonal one). Each (segment, value head) unit is one serial chain of chunks, so a call with
// few units (one long prompt as a single segment) leaves most SMs idle. When the units fill at most half of the SMs, every
// segment is cut into up to kMaxPieces chunk-aligned pieces that build in parallel as
// segments of their own; the pieces of a segment are then composed back into its entry, the
// composition the pages state for consecutive cached segments ("Cut First-Token Latency by
// 3.25x ..." (besthub.dev), paragraph "For linear layers": T_C2 S(C1) + S(C2), transition
// T_C2 T_C1) applied inside one segment. The decision depends on the current device's SM
// count; without a device there is no split.
constexpr int kMaxPieces = 8;

int gdn_split_m(const hypic_build_args *a) {
    const int64_t units = (int64_t)a->n_seg * a->H_v;
    if (units == 0 || a->O) return 1;   // a piece's outputs would need the state before it
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return 1;
    }
    if (2 * units > sms) return 1;
    return (int)std::min<int64_t>(kMaxPieces, sms / units);
}

// pieces of one segment of `len` tokens (1: built whole)
int seg_pieces(int64_t len, int m) {
    const int64_t nch = len > 0 ? (len + kGdnChunk - 1) / kGdnChunk : 0;
    return (int)std::max<int64_t>(1, std::min<int64_t>(m, nch));
}

// Workspace of the split: piece outputs S, P (dense families only) [slots][H_v][d][d] and lam
// [slots][H_v] ([slots][H_v][d] for diagonal gates). The pieces are composed straight into the
// outputs (the last state, the summed lam and, dense, the product).
//
// A second, narrower case: a DeltaNet / GDN call whose units take several rounds of SMs with
// a last round at most half full (16 segments x 32 heads on 152 SMs: 56 units in round four).
// Its trailing segments (the shortest, equal in length, last in the caller's order, outputs
// adjacent) are cut in two, so the last round runs half-length pieces, and all of their
// pieces are composed back in one batched launch (pieces laid out [piece][segment][head]).
struct SplitLayout {
    int m = 1, slots = 0, max_pieces = 1;
    int tail_first = -1, tail_count = 0;   // batched halving of segments [first, first + count)
    size_t off_S = 0, off_P = 0, off_lam = 0, bytes = 0;
    int pieces(const hypic_build_args *a, int j) const {
        if (tail_count > 0) return j >= tail_first && j < tail_first + tail_count ? 2 : 1;
        return m > 1 ? seg_pieces(a->seg_offsets[j + 1] - a->seg_offsets[j], m) : 1;
    }
};

// the trailing segments to halve, or 0 (see above)
int gdn_tail_split(const hypic_build_args *a, int *first) {
    if (!dense_family(a->family)) return 0;
    if (a->O) return 0;
    if (a->out_seg_stride != 0 && a->out_seg_stride != a->H_v) return 0;
    const int64_t units = (int64_t)a->n_seg * a->H_v;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    if (units <= sms) return 0;
    const int64_t last = units - ((units + sms - 1) / sms - 1) * sms;   // units of the last round
    if (2 * last > sms) return 0;
    const int cnt = (int)((last + a->H_v - 1) / a->H_v);
    if (cnt >= a->n_seg) return 0;
    const int j0 = a->n_seg - cnt;
    const int64_t len = a->seg_offsets[j0 + 1] - a->seg_offsets[j0];
    if ((len + kGdnChunk - 1) / kGdnChunk < 2) return 0;
    for (int j = 0; j < a->n_seg; ++j) {
        const int64_t lj = a->seg_offsets[j + 1] - a->seg_offsets[j];
        if (j >= j0 ? lj != len : lj < len) return 0;
    }
    *first = j0;
    return cnt;
}

SplitLayout gdn_split_layout(const hypic_build_args *a, size_t base) {
    SplitLayout L;
    L.m = gdn_split_m(a);
    if (L.m <= 1) {
        L.m = 1;
        L.tail_count = gdn_tail_split(a, &L.tail_first);
        if (L.tail_count == 0) return L;
        L.slots = 2 * L.tail_count;
        L.max_pieces = 2;
    } else {
        for (int j = 0; j < a->n_seg; ++j) {
            const int pj = seg_pieces(a->seg_offsets[j + 1] - a->seg_offsets[j], L.m);
            if (pj > 1) {
                L.slots += pj;
                L.max_pieces = std::max(L.max_pieces, pj);
            }
        }
        if (L.slots == 0) {
            L.m = 1;
            return L;
        }
    }
    const size_t unit = (size_t)a->d_k * a->d_k * sizeof(float);
    const size_t su = (size_t)L.slots * a->H_v;
    const bool dense = dense_family(a->family);
    const size_t nl = a->family == HYPIC_FAM_DIAG ? (size_t)a->d_k : 1;
    L.off_S = base;
    L.off_P = L.off_S + su * unit;
    L.off_lam = L.off_P + (dense ? su * unit : 0);
    L.bytes = L.off_lam + ((su * nl * sizeof(float) + 255) & ~(size_t)255) - base;
    return L;
}

bool build_shape_ok(const hypic_build_args *a) {
    return a && a->family >= HYPIC_FAM_LINEAR && a->family <= HYPIC_FAM_KDA &&
           (a->dtype == HYPIC_BF16 || a->dtype == HYPIC_F32) && a->n_seg >= 0 &&
           a->n_seg <= HYPIC_MAX_SEGMENTS && a->H_k > 0 && a->H_v > 0 && a->H_v % a->H_k == 0 &&
           head_size_ok(a->d_k, a->d_v);
}

bool compose_shape_ok(const hypic_compose_args *a) {
    return a && a->family >= HYPIC_FAM_LINEAR && a->family <= HYPIC_FAM_KDA && a->n_seg >= 0 &&
           a->n_units >= 0 && head_size_ok(a->d_k, a->d_v);
}

// The convolution-state warm-up's workspace: the heads' convolved k, v (fp32), their gathered
// gates and b, then the head entries of every (segment, value head) unit, built here (the
// composition reads the cached rests where the caller keeps them), and, for a dense scan that
// cannot write its last state directly (d < 128), the scan's prefix states.
struct WarmupLayout {
    int64_t rows = 0;
    size_t off_kh = 0, off_vh = 0, off_gh = 0, off_bh = 0, off_S = 0, off_lam = 0, off_P = 0, off_pre = 0,
           bytes = 0;
};

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

bool warmup_shape_ok(const hypic_warmup_args *a) {
    return a && a->family >= HYPIC_FAM_LINEAR && a->family <= HYPIC_FAM_KDA &&
           (a->dtype == HYPIC_BF16 || a->dtype == HYPIC_F32) && a->n_seg >= 0 &&
           a->n_seg <= HYPIC_MAX_SEGMENTS && a->H_k > 0 && a->H_v > 0 && a->H_v % a->H_k == 0 &&
           head_size_ok(a->d_k, a->d_v) && a->conv_k >= 1 && a->conv_k <= 8;
}

WarmupLayout warmup_layout(const hypic_warmup_args *a) {
    WarmupLayout L;
    for (int j = 0; j < a->n_seg; ++j)
        L.rows += std::max<int64_t>(0, std::min<int64_t>(a->conv_k - 1, a->seg_offsets[j + 1] - a->seg_offsets[j]));
    const size_t D = (size_t)a->d_k, U = (size_t)a->n_seg * a->H_v, R = (size_t)L.rows;
    const bool chan = a->family == HYPIC_FAM_DIAG || a->family == HYPIC_FAM_KDA;
    const bool dense = dense_family(a->family);
    L.off_vh = align256(R * a->H_k * D * 4);
    L.off_gh = L.off_vh + align256(R * a->H_v * D * 4);
    L.off_bh = L.off_gh + align256(a->log_gate ? R * a->H_v * (chan ? D : 1) * 4 : 0);
    L.off_S = L.off_bh + align256(a->beta ? R * a->H_v * 4 : 0);
    L.off_lam = L.off_S + align256(U * D * D * 4);
    L.off_P = L.off_lam + align256(U * (a->family == HYPIC_FAM_DIAG ? D : 1) * 4);
    L.off_pre = L.off_P + align256(dense ? U * D * D * 4 : 0);
    L.bytes = L.off_pre + align256(dense && D != 128 ? 2 * U * D * D * 4 : 0);
    return L;
}

}  // namespace

extern "C" {

int32_t hypic_abi_version(void) { return 5; }

const char *hypic_status_string(hypic_status s) {
    switch (s) {
    case HYPIC_OK: return "ok";
    case HYPIC_ERR_INVALID_ARG: return "invalid argument";
    case HYPIC_ERR_ALIGNMENT: return "misaligned tensor pointer";
    case HYPIC_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case HYPIC_ERR_RANGE: return "gate outside the supported range";
    case HYPIC_ERR_CUDA: return "CUDA runtime error";
    case HYPIC_ERR_TIMEOUT: return "device wait timed out";
    case HYPIC_ERR_BOUNDS: return "device index check failed";
    }
    return "unknown status";
}

size_t hypic_build_workspace_bytes(const hypic_build_args *a) {
    if (!build_shape_ok(a) || a->n_seg == 0 || !a->seg_offsets) return 0;
    const BuildPath path = pick_build(a);
    if (path == BuildPath::GatedTc) return gdn_split_layout(a, 0).bytes;   // 0 without a split
    if (path != BuildPath::GdnTc) return 0;
    if (gdn_records(a) == 0) return 0;
    const size_t base = gdn_records_bytes(a);
    return base + gdn_split_layout(a, base).bytes;
}

hypic_status hypic_build_segments(const hypic_build_args *a, void *stream) {
    NvtxRange range("hypic_build_segments");
    if (!a) return HYPIC_ERR_INVALID_ARG;
    const int fam = a->family;
    if (fam < HYPIC_FAM_LINEAR || fam > HYPIC_FAM_KDA) return HYPIC_ERR_INVALID_ARG;
    if (a->dtype != HYPIC_BF16 && a->dtype != HYPIC_F32) return HYPIC_ERR_INVALID_ARG;
    if (a->n_seg < 0 || a->n_seg > HYPIC_MAX_SEGMENTS) return HYPIC_ERR_INVALID_ARG;
    if (a->H_k <= 0 || a->H_v <= 0 || a->H_v % a->H_k != 0) return HYPIC_ERR_INVALID_ARG;
    if (a->d_k <= 0 || a->d_v <= 0) return HYPIC_ERR_INVALID_ARG;
    if (!head_size_ok(a->d_k, a->d_v)) return HYPIC_ERR_UNSUPPORTED;
    if (a->out_seg_stride < 0 || (a->out_seg_stride != 0 && a->out_seg_stride < a->H_v))
        return HYPIC_ERR_INVALID_ARG;
    if (a->n_seg == 0) return HYPIC_OK;
    if (!a->seg_offsets || a->seg_offsets[0] != 0) return HYPIC_ERR_INVALID_ARG;
    int max_len = 0;
    for (int j = 0; j < a->n_seg; ++j) {
        const int64_t len = a->seg_offsets[j + 1] - a->seg_offsets[j];
        if (len < 0) return HYPIC_ERR_INVALID_ARG;
        max_len = (int)std::min<int64_t>(std::max<int64_t>(max_len, len), INT32_MAX);
    }
    const int64_t n_tok = a->seg_offsets[a->n_seg];
    if (n_tok > INT32_MAX) return HYPIC_ERR_UNSUPPORTED;

    // required / forbidden tensors per family
    const bool delta = dense_family(fam);
    const bool need_gate = fam == HYPIC_FAM_DIAG || fam == HYPIC_FAM_GDN || fam == HYPIC_FAM_KDA;
    if (!a->S || !a->lam) return HYPIC_ERR_INVALID_ARG;
    if ((!a->q) != (!a->O)) return HYPIC_ERR_INVALID_ARG;   // queries exactly when outputs
    if (delta && (!a->P || !a->beta)) return HYPIC_ERR_INVALID_ARG;
    if (need_gate && !a->log_gate) return HYPIC_ERR_INVALID_ARG;
    if (fam == HYPIC_FAM_SCALAR && (!a->log_gate) == (!a->log_gamma)) return HYPIC_ERR_INVALID_ARG;
    if (n_tok > 0 && (!a->k || !a->v)) return HYPIC_ERR_INVALID_ARG;

    // alignment (16 B for tensors read or written with vector / bulk accesses)
    const void *v16[] = {a->k, a->v, a->S, a->P, a->q, a->O, a->S_init};
    for (const void *p : v16)
        if (p && !aligned(p, 16)) return HYPIC_ERR_ALIGNMENT;
    const void *v4[] = {a->log_gate, a->log_gamma, a->beta, a->lam};
    for (const void *p : v4)
        if (p && !aligned(p, 4)) return HYPIC_ERR_ALIGNMENT;

    // every tensor the kernels touch must be device memory of the current device
    const void *dev_ptrs[] = {a->S, a->lam, a->P, a->log_gamma, a->S_init};
    for (const void *p : dev_ptrs)
        if (p && !on_device(p)) return HYPIC_ERR_INVALID_ARG;
    if (n_tok > 0) {
        const void *in_ptrs[] = {a->k, a->v, a->log_gate, a->beta, a->q, a->O};
        for (const void *p : in_ptrs)
            if (p && !on_device(p)) return HYPIC_ERR_INVALID_ARG;
    }
    if (a->O && n_tok > 0) {   // the outputs overlap no input and no other output
        const size_t el = a->dtype == HYPIC_BF16 ? 2 : 4;
        const size_t nO = (size_t)n_tok * a->H_v * a->d_v * el;
        const size_t nk = (size_t)n_tok * a->H_k * a->d_k * el, nv = (size_t)n_tok * a->H_v * a->d_v * el;
        const int64_t stride = a->out_seg_stride ? a->out_seg_stride : a->H_v;
        const size_t units = (size_t)((a->n_seg - 1) * stride + a->H_v);
        const size_t nS = units * a->d_k * a->d_v * 4;
        const size_t nl = units * (fam == HYPIC_FAM_DIAG ? a->d_k : 1) * 4;
        if (overlaps(a->O, nO, a->k, nk) || overlaps(a->O, nO, a->v, nv) || overlaps(a->O, nO, a->q, nk) ||
            overlaps(a->O, nO, a->S, nS) || overlaps(a->O, nO, a->P, delta ? nS : 0) ||
            overlaps(a->O, nO, a->lam, nl))
            return HYPIC_ERR_INVALID_ARG;
    }
    const BuildPath path = pick_build(a);
    // records are addressed as 64-row blocks of a 2D tensor map with int32 coordinates
    if (path == BuildPath::GdnTc && gdn_records(a) > (int64_t)(INT32_MAX / 64)) return HYPIC_ERR_UNSUPPORTED;
    const size_t ws_need = hypic_build_workspace_bytes(a);
    if (ws_need > 0) {
        if (!a->workspace) return HYPIC_ERR_INVALID_ARG;
        if (!aligned(a->workspace, 16)) return HYPIC_ERR_ALIGNMENT;
        if (!on_device(a->workspace)) return HYPIC_ERR_INVALID_ARG;
    }
    if (ws_need > a->workspace_bytes) return HYPIC_ERR_INVALID_ARG;

    unsigned *err = status_word(nullptr);
    if (!err) return HYPIC_ERR_CUDA;

    static thread_local BuildParams p;   // ~12 KB: kept off the stack
    std::memset(&p, 0, sizeof(p));
    p.family = fam;
    p.dtype = a->dtype;
    p.n_seg = a->n_seg;
    p.H_k = a->H_k;
    p.H_v = a->H_v;
    p.D = a->d_k;
    p.gqa = a->H_v / a->H_k;
    p.max_len = max_len;
    p.n_tok = (int32_t)n_tok;
    p.seg_stride = a->out_seg_stride ? a->out_seg_stride : a->H_v;
    p.k = a->k;
    p.v = a->v;
    p.log_gate = a->log_gate;
    p.log_gamma = a->log_gamma;
    p.beta = a->beta;
    p.S = a->S;
    p.lam = a->lam;
    p.P = a->P;
    p.workspace = a->workspace;
    p.q = a->q;
    p.O = a->O;
    p.S_init = a->S_init;
    p.err = err;
    // the launch table: whole segments, or the chunk-aligned pieces of split ones (piece k of
    // a segment with n chunks in pj pieces covers chunks [k n / pj, (k + 1) n / pj))
    SplitLayout split;
    if (path == BuildPath::GdnTc || path == BuildPath::GatedTc) {
        const size_t base = path == BuildPath::GdnTc ? gdn_records_bytes(a) : 0;
        if (path == BuildPath::GdnTc && fam == HYPIC_FAM_KDA) {
            const size_t r = (size_t)gdn_records(a);
            uint8_t *x = static_cast<uint8_t *>(a->workspace) + r * (size_t)kGdnRecordBytes + (size_t)kGdnWorkspaceTail;
            p.kda_kt = x;
            p.kda_kh = x + r * (size_t)kKdaTileBytes;
            p.kda_side = reinterpret_cast<float *>(x + 2 * r * (size_t)kKdaTileBytes);
        }
        split = gdn_split_layout(a, base);
        if (split.slots > 0) {
            uint8_t *ws = static_cast<uint8_t *>(a->workspace);
            p.S_piece = reinterpret_cast<float *>(ws + split.off_S);
            p.P_piece = reinterpret_cast<float *>(ws + split.off_P);
            p.lam_piece = reinterpret_cast<float *>(ws + split.off_lam);
        }
    }
    std::vector<SegEntry> table;
    table.reserve(a->n_seg);
    int32_t slot = 0;
    for (int j = 0; j < a->n_seg; ++j) {
        const int64_t st = a->seg_offsets[j], len = a->seg_offsets[j + 1] - st;
        const int pj = split.pieces(a, j);
        if (pj == 1) {
            table.push_back(SegEntry{(int32_t)st, (int32_t)len, j, 0});
            continue;
        }
        const int64_t nch = (len + kGdnChunk - 1) / kGdnChunk;
        for (int k = 0; k < pj; ++k) {
            const int64_t t0 = (k * nch / pj) * kGdnChunk;
            const int64_t t1 = std::min<int64_t>(((k + 1) * nch / pj) * kGdnChunk, len);
            // batched tail halves: slot [piece][segment]; otherwise a segment's pieces in a row
            const int32_t sl = split.tail_count > 0 ? k * split.tail_count + (j - split.tail_first) : slot++;
            table.push_back(SegEntry{(int32_t)(st + t0), (int32_t)(t1 - t0), -1 - sl, 0});
        }
    }
    if ((int64_t)table.size() > HYPIC_MAX_SEGMENTS) return HYPIC_ERR_UNSUPPORTED;   // not reached: splits need few units
    std::stable_sort(table.begin(), table.end(), [](const SegEntry &x, const SegEntry &y) { return x.len > y.len; });
    p.n_seg = (int32_t)table.size();
    int64_t wsb = 0;
    for (int r = 0; r < p.n_seg; ++r) {
        p.seg[r] = table[r];
        p.seg[r].wsb = (int32_t)wsb;   // bounded by the record check above on the GDN path
        wsb = std::min<int64_t>(wsb + (int64_t)a->H_v * ((p.seg[r].len + kGdnChunk - 1) / kGdnChunk),
                                INT32_MAX);
    }

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    switch (path) {
    case BuildPath::GdnTc:
    case BuildPath::GatedTc: {
        cudaError_t e = path == BuildPath::GdnTc ? launch_build_gdn_tc(p, s) : launch_build_gated_tc(p, s);
        if (e != cudaSuccess || split.slots == 0) return from_cuda(e);
        // compose the pieces of every split segment into its entry: S = the pieces' prefix
        // scan from a zero state (its last state, copied out), lam = sum, P = product
        const bool dense = dense_family(fam);
        const size_t unit = (size_t)a->d_k * a->d_k;
        const size_t nl = fam == HYPIC_FAM_DIAG ? (size_t)a->d_k : 1;
        const int64_t stride = p.seg_stride;
        if (split.tail_count > 0) {   // one launch for all halved segments (adjacent outputs)
            const int64_t nu = (int64_t)split.tail_count * a->H_v;
            ComposeParams q;
            std::memset(&q, 0, sizeof(q));
            q.family = fam;
            q.n_seg = 2;
            q.n_units = nu;
            q.D = a->d_k;
            q.S = p.S_piece;
            q.lam = p.lam_piece;
            q.P = p.P_piece;
            q.prefix_last = a->S + (size_t)split.tail_first * a->H_v * unit;   // the segments' S
            q.lam_total = a->lam + (size_t)split.tail_first * a->H_v;
            q.P_total = a->P + (size_t)split.tail_first * a->H_v * unit;
            q.err = err;
            return from_cuda(launch_compose_dense_tc(q, s));
        }
        int32_t slot0 = 0;
        for (int j = 0; j < a->n_seg && e == cudaSuccess; ++j) {
            const int pj = split.pieces(a, j);
            if (pj == 1) continue;
            ComposeParams q;
            std::memset(&q, 0, sizeof(q));
            q.family = fam;
            q.n_seg = pj;
            q.n_units = a->H_v;
            q.D = a->d_k;
            q.S = p.S_piece + (size_t)slot0 * a->H_v * unit;
            q.lam = p.lam_piece + (size_t)slot0 * a->H_v * nl;
            q.P = dense ? p.P_piece + (size_t)slot0 * a->H_v * unit : nullptr;
            q.lam_total = a->lam + (size_t)j * stride * nl;
            q.P_total = dense ? a->P + (size_t)j * stride * unit : nullptr;
            q.err = err;
            // one launch: the last state straight into S, lam_total summed inside
            q.prefix_last = a->S + (size_t)j * stride * unit;
            e = dense ? launch_compose_dense_tc(q, s) : launch_compose_scaled(q, s);
            slot0 += pj;
        }
        return from_cuda(e);
    }
    case BuildPath::Seq: return from_cuda(launch_build_seq(p, s));
    case BuildPath::GatedSimt: return from_cuda(launch_build_gated_simt(p, s));
    case BuildPath::None: break;
    }
    return HYPIC_OK;
}

hypic_status hypic_build_segments_static_ws(const hypic_build_args *a, void *stream) {
    if (!a) return HYPIC_ERR_INVALID_ARG;
    const size_t need = hypic_build_workspace_bytes(a);
    if (need > (size_t)HYPIC_STATIC_WS_BYTES) return HYPIC_ERR_UNSUPPORTED;
    hypic_build_args b = *a;
    b.workspace = nullptr;
    b.workspace_bytes = 0;
    if (need) {
        void *ws = static_workspace();
        if (!ws) return HYPIC_ERR_CUDA;
        b.workspace = ws;
        b.workspace_bytes = (size_t)HYPIC_STATIC_WS_BYTES;
    }
    return hypic_build_segments(&b, stream);
}

hypic_status hypic_compose_scan(const hypic_compose_args *a, void *stream) {
    NvtxRange range("hypic_compose_scan");
    if (!a) return HYPIC_ERR_INVALID_ARG;
    const int fam = a->family;
    if (fam < HYPIC_FAM_LINEAR || fam > HYPIC_FAM_KDA) return HYPIC_ERR_INVALID_ARG;
    if (a->n_seg < 0 || a->n_units < 0) return HYPIC_ERR_INVALID_ARG;
    if (a->d_k <= 0 || a->d_v <= 0) return HYPIC_ERR_INVALID_ARG;
    if (!head_size_ok(a->d_k, a->d_v)) return HYPIC_ERR_UNSUPPORTED;
    if (a->n_seg == 0 || a->n_units == 0) return HYPIC_OK;
    if (a->n_units > (int64_t)INT32_MAX / 16) return HYPIC_ERR_UNSUPPORTED;
    const bool dense = dense_family(fam);
    if (!a->S || !a->prefix) return HYPIC_ERR_INVALID_ARG;
    if (fam != HYPIC_FAM_LINEAR && !a->lam) return HYPIC_ERR_INVALID_ARG;
    if (dense && !a->P) return HYPIC_ERR_INVALID_ARG;
    if (a->P_total && (!dense || !a->lam_total)) return HYPIC_ERR_INVALID_ARG;
    const void *v16[] = {a->S, a->P, a->S0, a->prefix, a->P_total};
    for (const void *p : v16)
        if (p && !aligned(p, 16)) return HYPIC_ERR_ALIGNMENT;
    if (a->lam && !aligned(a->lam, 4)) return HYPIC_ERR_ALIGNMENT;
    if (a->lam_total && !aligned(a->lam_total, 4)) return HYPIC_ERR_ALIGNMENT;
    const void *dev_ptrs[] = {a->S, a->P, a->S0, a->prefix, fam == HYPIC_FAM_LINEAR ? nullptr : a->lam,
                              a->lam_total, a->P_total};
    for (const void *p : dev_ptrs)
        if (p && !on_device(p)) return HYPIC_ERR_INVALID_ARG;

    const size_t D = (size_t)a->d_k;
    const size_t state_bytes = (size_t)a->n_seg * a->n_units * D * D * sizeof(float);
    const size_t lam_bytes = (size_t)a->n_seg * a->n_units * (fam == HYPIC_FAM_DIAG ? D : 1) * 4;
    if (overlaps(a->prefix, state_bytes, a->S, state_bytes) ||
        overlaps(a->prefix, state_bytes, a->P, dense ? state_bytes : 0) ||
        overlaps(a->prefix, state_bytes, a->lam, lam_bytes) ||
        overlaps(a->prefix, state_bytes, a->S0, (size_t)a->n_units * D * D * 4))
        return HYPIC_ERR_INVALID_ARG;
    // the totals overlap nothing: not the inputs, not prefix, not each other
    const size_t unit_bytes = (size_t)a->n_units * D * D * 4;
    const size_t lt_bytes = (size_t)a->n_units * (fam == HYPIC_FAM_DIAG ? D : 1) * 4;
    const struct { const void *p; size_t n; } ins[] = {
        {a->S, state_bytes}, {a->P, dense ? state_bytes : 0}, {a->lam, lam_bytes},
        {a->S0, unit_bytes}, {a->prefix, state_bytes}};
    for (const auto &in : ins)
        if (overlaps(a->lam_total, lt_bytes, in.p, in.n) || overlaps(a->P_total, unit_bytes, in.p, in.n))
            return HYPIC_ERR_INVALID_ARG;
    if (overlaps(a->lam_total, lt_bytes, a->P_total, unit_bytes)) return HYPIC_ERR_INVALID_ARG;

    unsigned *err = status_word(nullptr);
    if (!err) return HYPIC_ERR_CUDA;
    ComposeParams p;
    std::memset(&p, 0, sizeof(p));
    p.family = fam;
    p.n_seg = a->n_seg;
    p.n_units = a->n_units;
    p.D = a->d_k;
    p.S = a->S;
    p.lam = a->lam;
    p.P = a->P;
    p.S0 = a->S0;
    p.prefix = a->prefix;
    p.lam_total = a->lam_total;
    p.P_total = a->P_total;
    p.err = err;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    switch (pick_compose(a)) {
    case ComposePath::DenseTc: e = launch_compose_dense_tc(p, s); break;
    case ComposePath::DenseCols: e = launch_compose_dense_cols(p, s); break;
    case ComposePath::DenseSimt: e = launch_compose_dense_simt(p, s); break;
    case ComposePath::Scaled: e = launch_compose_scaled(p, s); break;
    case ComposePath::None: break;
    }
    // the dense tensor-core and the scaled kernels sum lam_total themselves (when they run)
    const ComposePath path = pick_compose(a);
    if (e == cudaSuccess && a->lam_total && path != ComposePath::DenseTc && path != ComposePath::Scaled)
        e = launch_compose_lam_total(p, s);
    return from_cuda(e);
}

hypic_status hypic_probe_wait_timeout(uint32_t limit_us, void *stream) {
    if (limit_us < 1 || limit_us > 1000000u) return HYPIC_ERR_INVALID_ARG;
    int dev = 0, sms = 0;
    unsigned *err = status_word(&dev);
    if (!err) return HYPIC_ERR_CUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        return HYPIC_ERR_CUDA;
    wait_probe_kernel<<<sms, 32, 0, static_cast<cudaStream_t>(stream)>>>(err, (uint64_t)limit_us * 1000u);
    return from_cuda(cudaGetLastError());
}

size_t hypic_warmup_workspace_bytes(const hypic_warmup_args *a) {
    if (!warmup_shape_ok(a) || a->n_seg == 0 || !a->seg_offsets) return 0;
    for (int j = 0; j < a->n_seg; ++j)
        if (a->seg_offsets[j + 1] < a->seg_offsets[j]) return 0;
    return warmup_layout(a).bytes;
}

hypic_status hypic_conv_warmup(const hypic_warmup_args *a, void *stream) {
    NvtxRange range("hypic_conv_warmup");
    if (!a) return HYPIC_ERR_INVALID_ARG;
    const int fam = a->family;
    if (fam < HYPIC_FAM_LINEAR || fam > HYPIC_FAM_KDA) return HYPIC_ERR_INVALID_ARG;
    if (a->dtype != HYPIC_BF16 && a->dtype != HYPIC_F32) return HYPIC_ERR_INVALID_ARG;
    if (a->n_seg < 0 || a->n_seg > HYPIC_MAX_SEGMENTS) return HYPIC_ERR_INVALID_ARG;
    if (a->H_k <= 0 || a->H_v <= 0 || a->H_v % a->H_k != 0) return HYPIC_ERR_INVALID_ARG;
    if (a->d_k <= 0 || a->d_v <= 0) return HYPIC_ERR_INVALID_ARG;
    if (a->conv_k < 1 || a->conv_k > 8) return HYPIC_ERR_INVALID_ARG;
    if (!head_size_ok(a->d_k, a->d_v)) return HYPIC_ERR_UNSUPPORTED;
    if (a->n_seg == 0) return HYPIC_OK;
    if (!a->seg_offsets || a->seg_offsets[0] != 0) return HYPIC_ERR_INVALID_ARG;
    for (int j = 0; j < a->n_seg; ++j)
        if (a->seg_offsets[j + 1] < a->seg_offsets[j]) return HYPIC_ERR_INVALID_ARG;
    const int64_t n_tok = a->seg_offsets[a->n_seg];
    if (n_tok > INT32_MAX) return HYPIC_ERR_UNSUPPORTED;
    const bool dense = dense_family(fam);
    const bool need_gate = fam == HYPIC_FAM_DIAG || fam == HYPIC_FAM_GDN || fam == HYPIC_FAM_KDA;
    if (!a->S_rest || !a->lam_rest || !a->S || !a->lam || !a->conv_wk || !a->conv_wv) return HYPIC_ERR_INVALID_ARG;
    if (dense && (!a->P_rest || !a->P || !a->beta)) return HYPIC_ERR_INVALID_ARG;
    if (need_gate && !a->log_gate) return HYPIC_ERR_INVALID_ARG;
    if (fam == HYPIC_FAM_SCALAR && (!a->log_gate) == (!a->log_gamma)) return HYPIC_ERR_INVALID_ARG;
    if (n_tok > 0 && (!a->k_raw || !a->v_raw)) return HYPIC_ERR_INVALID_ARG;
    const void *v16[] = {a->k_raw, a->v_raw, a->S_rest, a->P_rest, a->S, a->P};
    for (const void *p : v16)
        if (p && !aligned(p, 16)) return HYPIC_ERR_ALIGNMENT;
    const void *v4[] = {a->conv_wk, a->conv_wv, a->log_gate, a->log_gamma, a->beta, a->lam_rest, a->lam};
    for (const void *p : v4)
        if (p && !aligned(p, 4)) return HYPIC_ERR_ALIGNMENT;
    const void *dev[] = {a->conv_wk, a->conv_wv, a->log_gamma, a->S_rest, a->lam_rest, a->P_rest,
                         a->S, a->lam, a->P};
    for (const void *p : dev)
        if (p && !on_device(p)) return HYPIC_ERR_INVALID_ARG;
    if (n_tok > 0) {
        const void *in[] = {a->k_raw, a->v_raw, a->log_gate, a->beta};
        for (const void *p : in)
            if (p && !on_device(p)) return HYPIC_ERR_INVALID_ARG;
    }
    // the outputs overlap no input and no other output
    const size_t D = (size_t)a->d_k, U = (size_t)a->n_seg * a->H_v, el = a->dtype == HYPIC_BF16 ? 2 : 4;
    const bool chan = fam == HYPIC_FAM_DIAG || fam == HYPIC_FAM_KDA;
    const size_t nS = U * D * D * 4, nl = U * (fam == HYPIC_FAM_DIAG ? D : 1) * 4;
    const struct { const void *p; size_t n; } ins[] = {
        {a->k_raw, (size_t)n_tok * a->H_k * D * el}, {a->v_raw, (size_t)n_tok * a->H_v * D * el},
        {a->conv_wk, (size_t)a->H_k * D * a->conv_k * 4}, {a->conv_wv, (size_t)a->H_v * D * a->conv_k * 4},
        {a->log_gate, (size_t)n_tok * a->H_v * (chan ? D : 1) * 4}, {a->log_gamma, (size_t)a->H_v * 4},
        {a->beta, (size_t)n_tok * a->H_v * 4}, {a->S_rest, nS}, {a->lam_rest, nl}, {a->P_rest, dense ? nS : 0}};
    const struct { const void *p; size_t n; } outs[] = {{a->S, nS}, {a->lam, nl}, {a->P, dense ? nS : 0}};
    for (const auto &o : outs) {
        for (const auto &i : ins)
            if (overlaps(o.p, o.n, i.p, i.n)) return HYPIC_ERR_INVALID_ARG;
        for (const auto &o2 : outs)
            if (&o != &o2 && overlaps(o.p, o.n, o2.p, o2.n)) return HYPIC_ERR_INVALID_ARG;
    }
    const WarmupLayout L = warmup_layout(a);
    if (!a->workspace) return HYPIC_ERR_INVALID_ARG;
    if (!aligned(a->workspace, 16)) return HYPIC_ERR_ALIGNMENT;
    if (!on_device(a->workspace)) return HYPIC_ERR_INVALID_ARG;
    if (L.bytes > a->workspace_bytes) return HYPIC_ERR_INVALID_ARG;
    unsigned *err = status_word(nullptr);
    if (!err) return HYPIC_ERR_CUDA;
    uint8_t *ws = static_cast<uint8_t *>(a->workspace);
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    // (1) the heads' tokens convolved over the prompt's raw stream, with their gates and b
    static thread_local ConvHeadParams cp;   // ~8 KB: kept off the stack
    std::memset(&cp, 0, sizeof(cp));
    std::vector<int64_t> head_offs(a->n_seg + 1, 0);
    for (int j = 0; j < a->n_seg; ++j) {
        const int64_t hl = std::min<int64_t>(a->conv_k - 1, a->seg_offsets[j + 1] - a->seg_offsets[j]);
        cp.seg_start[j] = (int32_t)a->seg_offsets[j];
        cp.head_off[j] = (int32_t)head_offs[j];
        head_offs[j + 1] = head_offs[j] + hl;
    }
    cp.head_off[a->n_seg] = (int32_t)head_offs[a->n_seg];
    cp.family = fam;
    cp.dtype = a->dtype;
    cp.n_seg = a->n_seg;
    cp.H_k = a->H_k;
    cp.H_v = a->H_v;
    cp.D = a->d_k;
    cp.K = a->conv_k;
    cp.n_rows = (int32_t)L.rows;
    cp.k_raw = a->k_raw;
    cp.v_raw = a->v_raw;
    cp.wk = a->conv_wk;
    cp.wv = a->conv_wv;
    cp.log_gate = a->log_gate;
    cp.beta = a->beta;
    cp.k_head = reinterpret_cast<float *>(ws + L.off_kh);
    cp.v_head = reinterpret_cast<float *>(ws + L.off_vh);
    cp.g_head = a->log_gate ? reinterpret_cast<float *>(ws + L.off_gh) : nullptr;
    cp.b_head = a->beta ? reinterpret_cast<float *>(ws + L.off_bh) : nullptr;
    cp.err = err;
    cudaError_t e = launch_conv_heads(cp, s);
    if (e != cudaSuccess) return HYPIC_ERR_CUDA;

    // (2) the heads' entries from a zero state (fp32 inputs: the exact path, no workspace),
    //     into the first composition piece
    float *Sp = reinterpret_cast<float *>(ws + L.off_S);
    float *lp = reinterpret_cast<float *>(ws + L.off_lam);
    float *Pp = dense ? reinterpret_cast<float *>(ws + L.off_P) : nullptr;
    hypic_build_args b;
    std::memset(&b, 0, sizeof(b));
    b.family = fam;
    b.dtype = HYPIC_F32;
    b.n_seg = a->n_seg;
    b.H_k = a->H_k;
    b.H_v = a->H_v;
    b.d_k = a->d_k;
    b.d_v = a->d_v;
    b.seg_offsets = head_offs.data();
    b.k = cp.k_head;
    b.v = cp.v_head;
    b.log_gate = cp.g_head;
    b.log_gamma = a->log_gamma;
    b.beta = cp.b_head;
    b.S = Sp;
    b.lam = lp;
    b.P = Pp;
    const hypic_status st = hypic_build_segments(&b, stream);
    if (st != HYPIC_OK) return st;

    // (3) one composition of the head entries (segment 0) with the cached rests (segment 1, read
    //     where the caller keeps them): the last state (S), the summed lam and, dense, the
    //     product P_rest P_head
    ComposeParams q;
    std::memset(&q, 0, sizeof(q));
    q.family = fam;
    q.n_seg = 2;
    q.n_units = (int64_t)U;
    q.D = a->d_k;
    q.S = Sp;
    q.lam = lp;
    q.P = Pp;
    q.S1 = a->S_rest;
    q.lam1 = a->lam_rest;
    q.P1 = dense ? a->P_rest : nullptr;
    q.lam_total = a->lam;
    q.P_total = dense ? a->P : nullptr;
    q.err = err;
    if (!dense) {
        q.prefix_last = a->S;
        e = launch_compose_scaled(q, s);
    } else if (compose_dense_tc_supported(q)) {
        q.prefix_last = a->S;
        e = launch_compose_dense_tc(q, s);
    } else {
        float *pre = reinterpret_cast<float *>(ws + L.off_pre);
        q.prefix = pre;
        e = launch_compose_dense_simt(q, s);
        if (e == cudaSuccess) e = launch_compose_lam_total(q, s);
        if (e == cudaSuccess) e = cudaMemcpyAsync(a->S, pre + U * D * D, nS, cudaMemcpyDeviceToDevice, s);
    }
    return from_cuda(e);
}

const char *hypic_build_kernel_name(const hypic_build_args *a) {
    if (!build_shape_ok(a)) return nullptr;
    switch (pick_build(a)) {
    case BuildPath::GdnTc: return a->family == HYPIC_FAM_KDA ? "build_kda_tc" : "build_gdn_tc";
    case BuildPath::Seq: return "build_seq";
    case BuildPath::GatedTc: return "build_gated_tc";
    case BuildPath::GatedSimt: return "build_gated_simt";
    case BuildPath::None: break;
    }
    return "none";
}

const char *hypic_compose_kernel_name(const hypic_compose_args *a) {
    if (!compose_shape_ok(a)) return nullptr;
    switch (pick_compose(a)) {
    case ComposePath::DenseTc: return "compose_dense_tc";
    case ComposePath::DenseCols: return "compose_dense_cols";
    case ComposePath::DenseSimt: return "compose_dense_simt";
    case ComposePath::Scaled: return "compose_scaled";
    case ComposePath::None: break;
    }
    return "none";
}

hypic_status hypic_get_device_status(void *stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return HYPIC_ERR_CUDA;
    unsigned *w = status_word(nullptr);
    if (!w) return HYPIC_ERR_CUDA;
    unsigned v = 0;
    if (cudaMemcpy(&v, w, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return HYPIC_ERR_CUDA;
    if (v) {
        const unsigned zero = 0;
        if (cudaMemcpy(w, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
            return HYPIC_ERR_CUDA;
    }
    if (v & kErrBounds) return HYPIC_ERR_BOUNDS;
    if (v & kErrTimeout) return HYPIC_ERR_TIMEOUT;
    if (v & kErrRange) return HYPIC_ERR_RANGE;
    return HYPIC_OK;
}

}  // extern "C"
