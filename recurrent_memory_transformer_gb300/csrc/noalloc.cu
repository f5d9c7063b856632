// Segment attention for callers that cannot allocate device memory.
//
// armt_segment_attention_bf16 needs the values transposed into a caller
// buffer and allocates a small device error word on first use.  Some callers
// cannot do either: a serving process whose device memory is entirely owned
// by its own arena or memory cap, or a latency-critical path that must not
// hit cudaMalloc's implicit device-wide synchronisation.  This entry point
// takes q|k|v in the plain fused row layout and keeps all of its scratch --
// the transposed values and the error word -- in one file-scope device array
// of fixed size, so it calls no allocator at all.  A bounded wait inside the
// attention kernel that gives up records a code in that error word, which
// stays set (later calls see it too) until armt_noalloc_sync_status reads
// and clears it.
#include <cuda.h>
#include <cuda_runtime.h>

#include <string>

#include "../../include/armt.h"
#include "attn_tc.cuh"
#include "common.cuh"

using namespace armt;

namespace armt {
bool encode_tmap_bf16_3d(CUtensorMap* map, const void* base, int K, int rows, int layers,
                         int box_rows);
void set_last_error(const std::string& msg);  // text returned by armt_last_error()
void* current_context();                      // the calling thread's driver context
}

// Scratch shared by every call in the process on a given device: 256 bytes
// for the error word, then the transposed values.  Held by every GPU that
// loads the library until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[ARMT_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr size_t kErrBytes = 256;
constexpr int kMaxDevices = 64;
// Device address of g_noalloc_scratch per device, and the context it was
// looked up in: a new context (e.g. after cudaDeviceReset) reloads the
// module, so the address is looked up again.
struct ScratchAddr {
  std::atomic<void*> ctx{nullptr};
  std::atomic<unsigned char*> base{nullptr};
};
ScratchAddr g_scratch_addr[kMaxDevices];

armt_status nfail(armt_status s, const std::string& msg) {
  set_last_error(msg);
  return s;
}

// Device address of the scratch array on the current device.  Set-up, the
// first time on a device (or context): cudaGetSymbolAddress with the device
// current, and the error word cleared.  Allocates nothing.
armt_status scratch_base(unsigned char** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return nfail(ARMT_ERR_NO_DEVICE, "no current CUDA device");
  }
  void* ctx = current_context();
  ScratchAddr& a = g_scratch_addr[dev];
  unsigned char* base = a.base.load();
  if (base == nullptr || a.ctx.load() != ctx) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return nfail(ARMT_ERR_CUDA, std::string("cudaGetSymbolAddress: ") + cudaGetErrorString(e));
    }
    e = cudaMemset(p, 0, sizeof(int));  // the error word starts clear
    if (e != cudaSuccess) return nfail(ARMT_ERR_CUDA, std::string("cudaMemset: ") + cudaGetErrorString(e));
    base = static_cast<unsigned char*>(p);
    a.base.store(base);
    a.ctx.store(ctx);
  }
  *out = base;
  return ARMT_OK;
}

// vt[g][kvh][c][t] = qkv[g][t][(Hq + Hkv + kvh) * hd + c] for t < T, 0 for
// T <= t < t_pad.  One block per (t tile of 32, kv head, cell).
__global__ void transpose_v_kernel(const bf16* __restrict__ qkv, bf16* __restrict__ vt, int T,
                                   int t_pad, int Hq, int Hkv, int hd) {
  __shared__ bf16 tile[32][129];
  const int t0 = blockIdx.x * 32, kvh = blockIdx.y, g = blockIdx.z;
  const int ld = (Hq + 2 * Hkv) * hd;
  const bf16* src = qkv + (long long)g * T * ld + (long long)(Hq + Hkv + kvh) * hd;
  for (int i = threadIdx.x; i < 32 * hd; i += blockDim.x) {
    const int tt = i / hd, c = i - tt * hd;
    const int t = t0 + tt;
    tile[tt][c] = t < T ? src[(long long)t * ld + c] : __float2bfloat16_rn(0.f);
  }
  __syncthreads();
  bf16* dst = vt + ((long long)g * Hkv + kvh) * hd * t_pad;
  for (int i = threadIdx.x; i < 32 * hd; i += blockDim.x) {
    const int c = i / 32, tt = i - c * 32;
    const int t = t0 + tt;
    if (t < t_pad) dst[(long long)c * t_pad + t] = tile[tt][c];
  }
}

}  // namespace

extern "C" ARMT_API armt_status armt_segment_attention_bf16_noalloc(const void* qkv, void* out,
                                                                    int32_t G, int32_t T,
                                                                    int32_t Hq, int32_t Hkv,
                                                                    int32_t hd, void* stream) {
  if (qkv == nullptr || out == nullptr) return nfail(ARMT_ERR_ARG, "NULL argument");
  if (G <= 0 || T <= 0 || Hq <= 0 || Hkv <= 0) return nfail(ARMT_ERR_ARG, "sizes must be positive");
  if (Hq % Hkv != 0) return nfail(ARMT_ERR_SHAPE, "Hq must be a multiple of Hkv");
  if (hd != 64 && hd != 128) return nfail(ARMT_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
  if ((reinterpret_cast<uintptr_t>(qkv) | reinterpret_cast<uintptr_t>(out)) & 15)
    return nfail(ARMT_ERR_ARG, "pointers must be 16-byte aligned");
  const long long t_pad = (T + 7) / 8 * 8;
  const long long vt_bytes = (long long)G * Hkv * hd * t_pad * 2;
  if (vt_bytes + (long long)kErrBytes > (long long)ARMT_NOALLOC_SCRATCH_BYTES)
    return nfail(ARMT_ERR_SHAPE, "G * Hkv * hd * round_up(T, 8) * 2 = " + std::to_string(vt_bytes) +
                                     " bytes exceeds the fixed scratch of " +
                                     std::to_string((long long)ARMT_NOALLOC_SCRATCH_BYTES - (long long)kErrBytes) +
                                     " bytes");
  int dev = 0, nsm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return nfail(ARMT_ERR_NO_DEVICE, "no current CUDA device");
  }
  if (cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || nsm <= 0) {
    cudaGetLastError();
    return nfail(ARMT_ERR_CUDA, "multiprocessor count query failed");
  }
  // The array's name is only a host-side stand-in; kernels get this address.
  unsigned char* base = nullptr;
  {
    const armt_status sb = scratch_base(&base);
    if (sb != ARMT_OK) return sb;
  }
  int* err = reinterpret_cast<int*>(base);
  bf16* vt = reinterpret_cast<bf16*>(base + kErrBytes);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  transpose_v_kernel<<<dim3((unsigned)((t_pad + 31) / 32), (unsigned)Hkv, (unsigned)G), 256, 0, st>>>(
      reinterpret_cast<const bf16*>(qkv), vt, T, (int)t_pad, Hq, Hkv, hd);
  e = cudaGetLastError();
  if (e != cudaSuccess) return nfail(ARMT_ERR_CUDA, std::string("transpose: ") + cudaGetErrorString(e));
  CUtensorMap tq, tv;
  if (!encode_tmap_bf16_3d(&tq, qkv, (Hq + 2 * Hkv) * hd, T, G, 128) ||
      !encode_tmap_bf16_3d(&tv, vt, (int)t_pad, hd, G * Hkv, hd))
    return nfail(ARMT_ERR_CUDA, "cuTensorMapEncodeTiled failed");
  AttnArgs aa;
  aa.out = reinterpret_cast<bf16*>(out);
  aa.T = T;
  aa.Hq = Hq;
  aa.Hkv = Hkv;
  aa.g_first = 0;
  aa.n_qtiles = (T + 127) / 128;
  aa.scale_log2 = 1.4426950408889634f / sqrtf((float)hd);
  aa.err = err;
  aa.wp = wait_policy_from_env();
  e = hd == 64 ? launch_attn_tc<64>(tq, tv, aa, G, nsm, st) : launch_attn_tc<128>(tq, tv, aa, G, nsm, st);
  if (e != cudaSuccess) return nfail(ARMT_ERR_CUDA, std::string("attention: ") + cudaGetErrorString(e));
  return ARMT_OK;
}

// Waits for `stream`, then reports (ARMT_ERR_TIMEOUT) and clears a timeout
// that the no-allocation attention recorded on the current device since the
// last call.  Allocates nothing.
extern "C" ARMT_API armt_status armt_noalloc_sync_status(void* stream) {
  unsigned char* base = nullptr;
  {
    const armt_status sb = scratch_base(&base);
    if (sb != ARMT_OK) return sb;
  }
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return nfail(ARMT_ERR_CUDA, std::string("cudaStreamSynchronize: ") + cudaGetErrorString(e));
  int h = 0;
  e = cudaMemcpy(&h, base, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return nfail(ARMT_ERR_CUDA, std::string("cudaMemcpy: ") + cudaGetErrorString(e));
  if (h != 0) {
    e = cudaMemset(base, 0, sizeof(int));
    if (e != cudaSuccess) return nfail(ARMT_ERR_CUDA, std::string("cudaMemset: ") + cudaGetErrorString(e));
    return nfail(ARMT_ERR_TIMEOUT, "device wait timed out (code " + std::to_string(h) + ")");
  }
  return ARMT_OK;
}
