// kv_append.cuh -- fused K/V-cache append: the f32 K and V rows of T new
// tokens per sequence, rounded to the cache's 16-bit type (round to nearest
// even), written at cache row positions[b][t].  This is the step before the
// attention of a chunked prefill (minfer "11 · P5 — prefill gap session: TM=128
// big tiles + FA rewrite", section 3.2, the store_kv kernel: one f32 token row
// in, one 16-bit cache row out at the token's position), done here for K and V
// in one launch.
//
// The work is pure streaming (48 bytes of HBM traffic per 8 elements: 2 x 16 B
// of f32 read, 16 B of 16-bit written), so the kernel is shaped for HBM: every
// thread moves one 8-element group with two 16-byte streaming loads and one
// 16-byte store, consecutive threads take consecutive groups of a row (whole
// 128-byte lines on both sides), and a grid-stride loop runs over a grid of
// 8 CTAs of 256 threads per SM.
//
// Included by fa_prefill.cu (one translation unit: the kernel reports bad
// positions through the same device status word as the attention kernels).

namespace fa {

constexpr uint32_t WD_APPEND_POSITION = 32;  // status code: a position outside [0, kv_cap)
constexpr int APPEND_THREADS = 256;
constexpr int APPEND_CTAS_PER_SM = 8;

template <bool BF16>
__global__ void __launch_bounds__(APPEND_THREADS)
    kv_append_kernel(const float4* __restrict__ k_new, const float4* __restrict__ v_new,
                     const int* __restrict__ positions, uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                     int BT, int T, int groups, int cap) {
  // item i: group g = i % groups of row i / groups; rows [0, BT) are K, [BT, 2 BT) are V
  const int total = 2 * BT * groups;
  ptx::griddep_launch_dependents();
  ptx::griddep_wait();  // the previous kernel (e.g. the K/V projection) has completed
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
    const int row = i / groups;
    const int g = i - row * groups;
    const bool is_v = row >= BT;
    const int bt = is_v ? row - BT : row;
    const int pos = __ldg(positions + bt);
    if (pos < 0 || pos >= cap) {  // skipped and reported, never written
      const uint32_t at = bt < 0xFFFFFF ? static_cast<uint32_t>(bt) : 0xFFFFFFu;
      atomicCAS(&g_fa_status, 0u, WD_APPEND_POSITION | (at << 8));
      continue;
    }
    const float4* src = (is_v ? v_new : k_new) + (static_cast<size_t>(bt) * groups + g) * 2;
    const float4 a = __ldcs(src);
    const float4 b = __ldcs(src + 1);
    uint4 out;
    out.x = pack2<BF16>(a.x, a.y);
    out.y = pack2<BF16>(a.z, a.w);
    out.z = pack2<BF16>(b.x, b.y);
    out.w = pack2<BF16>(b.z, b.w);
    const int bb = bt / T;
    (is_v ? v_cache : k_cache)[(static_cast<size_t>(bb) * cap + pos) * groups + g] = out;
  }
}

// Host side: argument checks (no device call), then one launch.
static int run_kv_append(const void* k_new, const void* v_new, const void* positions, void* k_cache, void* v_cache,
                         int B, int T, int Hkv, int hd, int cap, bool bf16, void* stream) {
  if (B < 0 || T < 0 || Hkv < 1 || cap < 1) return FA_ERR_INVALID_ARG;
  if (hd < 8 || hd % 8 != 0) return FA_ERR_UNSUPPORTED;
  if (B == 0 || T == 0) return FA_OK;  // nothing to append; no pointer is read
  if (!k_new || !v_new || !positions || !k_cache || !v_cache) return FA_ERR_INVALID_ARG;
  const auto mis = [](const void* x, uintptr_t a) { return (reinterpret_cast<uintptr_t>(x) & (a - 1)) != 0; };
  if (mis(k_new, 16) || mis(v_new, 16) || mis(k_cache, 16) || mis(v_cache, 16) || mis(positions, 4))
    return FA_ERR_ALIGNMENT;
  const long long groups = (long long)Hkv * hd / 8;
  const long long bt = (long long)B * T;
  if (2 * bt * groups > 0x7FFFFFFFLL - (1LL << 22)) return FA_ERR_UNSUPPORTED;  // 32-bit item index, stride headroom
  const size_t new_bytes = (size_t)bt * groups * 32, cache_bytes = (size_t)B * cap * groups * 16;
  if (overlaps(k_cache, cache_bytes, v_cache, cache_bytes) || overlaps(k_cache, cache_bytes, k_new, new_bytes) ||
      overlaps(k_cache, cache_bytes, v_new, new_bytes) || overlaps(v_cache, cache_bytes, k_new, new_bytes) ||
      overlaps(v_cache, cache_bytes, v_new, new_bytes) || overlaps(k_cache, cache_bytes, positions, bt * 4) ||
      overlaps(v_cache, cache_bytes, positions, bt * 4))
    return FA_ERR_INVALID_ARG;
  int dev = -1;
  const int ds = check_device(&dev);
  if (ds != FA_OK) return ds;
  const long long items = 2 * bt * groups;
  const long long want = (items + APPEND_THREADS - 1) / APPEND_THREADS;
  const long long cap_ctas = (long long)g_dev_sms[dev].load() * APPEND_CTAS_PER_SM;
  const unsigned grid = static_cast<unsigned>(want < cap_ctas ? want : cap_ctas);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const float4* kn = static_cast<const float4*>(k_new);
  const float4* vn = static_cast<const float4*>(v_new);
  const int* ps = static_cast<const int*>(positions);
  uint4* kc = static_cast<uint4*>(k_cache);
  uint4* vc = static_cast<uint4*>(v_cache);
  const int bti = static_cast<int>(bt), gi = static_cast<int>(groups);
  const cudaError_t e =
      bf16 ? launch_pdl(kv_append_kernel<true>, dim3(grid), dim3(APPEND_THREADS), 0, st, kn, vn, ps, kc, vc, bti, T, gi, cap)
           : launch_pdl(kv_append_kernel<false>, dim3(grid), dim3(APPEND_THREADS), 0, st, kn, vn, ps, kc, vc, bti, T, gi,
                        cap);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return FA_ERR_LAUNCH;
  }
  return FA_OK;
}

}  // namespace fa
