// compact.cu -- step a4, ragged packing of the rows the target must score.
//
// "DFlash to DSpark in SGLang", section "Ragged verify under full CUDA
// graphs": the scheduled verify tokens are front-packed into one buffer and a
// cu_seqlens-style offset array marks where each request's segment starts.
// Request b owns rows row_off[b] + j, j = 0..L_b: the root token (j = 0, the
// last committed token, whose target row scores draft 1) and drafts
// d_1..d_{L_b}.  Its position is the cached length plus j.
//
// One thread per slot of the B*(gamma+1) capacity: slot (b, j) writes packed
// row row_off[b] + j when j <= L_b; slot t >= N_rows also writes the padding
// of row t.  The two write sets are disjoint.
#include "dspark_internal.cuh"

namespace dspark {
namespace {

__global__ void __launch_bounds__(kThreads) compact_kernel(const CompactArgs a) {
    // Launched as a programmatic dependent of the kernel before it on the
    // stream: wait here until that grid has completed and its writes (L,
    // row_off) are visible.  Without such a grid this returns at once.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // The verify that follows may be scheduled now (it waits for this grid).
    asm volatile("griddepcontrol.launch_dependents;");
    const int g1 = a.gamma + 1;
    const int cap = a.B * g1;
    const int t = blockIdx.x * kThreads + threadIdx.x;
    if (t >= cap) return;
    const int n_rows = a.row_off[a.B];
    const int b = t / g1, j = t - b * g1;
    const int r = a.row_off[b] + j;
    if (j <= a.L[b] && r >= 0 && r < cap) {
        int id;
        if (j == 0) id = a.last_tokens ? a.last_tokens[b] : -1;
        else id = a.draft_tokens[size_t(b) * a.gamma + j - 1];
        a.packed_ids[r] = id;
        a.packed_pos[r] = (a.seq_lens ? a.seq_lens[b] : 0) + j;
        a.row_req[r] = b;
        a.row_k[r] = j;
    }
    if (t >= n_rows) {
        a.packed_ids[t] = -1;
        a.packed_pos[t] = 0;
        a.row_req[t] = -1;
        a.row_k[t] = -1;
    }
}

}  // namespace

cudaError_t launch_compact(const CompactArgs &a, cudaStream_t s) {
    // Programmatic dependent launch: the grid is scheduled while the kernel
    // before it (the score kernel) still runs, so its launch latency is
    // hidden; griddepcontrol.wait above keeps the data dependency.
    const int cap = a.B * (a.gamma + 1);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((cap + kThreads - 1) / kThreads);
    cfg.blockDim = dim3(kThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, compact_kernel, a);
}

}  // namespace dspark
