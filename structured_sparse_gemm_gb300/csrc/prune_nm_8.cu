// prune_nm_8.cu -- N:M prune into 2:4 forms for the 8-bit element types.
#include "prune_nm.cuh"

namespace st24 {
namespace prune {

bool launch_nm_8bit(int dt, int n, int m, bool two, const void* W, int64_t M, int64_t K, int64_t ldw, void* values,
                    void* meta, int num_sms, cudaStream_t stream) {
  if (dt == kE4M3) return launch_nm<kE4M3, 1>(n, m, two, W, M, K, ldw, values, meta, num_sms, stream);
  if (dt == kS8) return launch_nm<kS8, 1>(n, m, two, W, M, K, ldw, values, meta, num_sms, stream);
  return false;
}

}  // namespace prune
}  // namespace st24
