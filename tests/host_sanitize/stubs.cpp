// Stand-ins for the CUDA launchers of the library, for a CPU-only build of
// the host layer under AddressSanitizer and UndefinedBehaviorSanitizer.  The
// paths the sanitizer driver exercises (configuration checks, buffer sizes,
// the decode work-item plan, failure injection, context creation failing
// before any kernel) never reach a launch; if one did, it would report "no
// device" instead of running anything.
#include "../../paged_kv_cache_flash_gb300/csrc/kvs_launch.h"

namespace kvs {

cudaError_t launch_append_step(const Geo &, const uint16_t *, const uint16_t *, uint16_t *, int32_t *,
                               kvs_record *, uint8_t *, const StepAppend *, const StepAppend *, uint32_t,
                               uint32_t, uint64_t, cudaStream_t) { return cudaErrorNoDevice; }
cudaError_t launch_append(const Geo &, const AppendArgs &, cudaStream_t) { return cudaErrorNoDevice; }
cudaError_t launch_decode(const Geo &, const CUtensorMap &, const Work &, const uint16_t *, const int32_t *,
                          uint32_t, uint32_t, int, cudaStream_t) { return cudaErrorNoDevice; }
cudaError_t launch_combine(const Geo &, const Work &, float *, uint32_t, uint32_t, uint32_t, uint32_t, cudaStream_t)
{ return cudaErrorNoDevice; }
cudaError_t launch_mass(const Geo &, const Work &, float *, uint32_t, kvs_record *, const ScoreArgs *, cudaStream_t)
{ return cudaErrorNoDevice; }
cudaError_t launch_score(const Geo &, const Work &, kvs_record *, const float *, double, uint32_t, double,
                         double, double, double, double, uint32_t, cudaStream_t) { return cudaErrorNoDevice; }
cudaError_t launch_radix_select(const Geo &, const Work &, const kvs_record *, uint32_t, uint32_t, int, double,
                                cudaStream_t) { return cudaErrorNoDevice; }
cudaError_t launch_select(const Geo &, const Work &, const kvs_record *, const int32_t *, int, double, uint32_t,
                          bool, const SelectOut &, cudaStream_t) { return cudaErrorNoDevice; }
uint32_t select_launches(uint32_t) { return 0; }
bool select_plan_fits(uint32_t) { return false; }
cudaError_t launch_select_plan(const Geo &, const Work &, const kvs_record *, const int32_t *, int, double, uint32_t,
                               uint32_t, const SelectOut &, cudaStream_t) { return cudaErrorNoDevice; }
cudaError_t launch_plan(const Work &, uint32_t, const SelectOut &, cudaStream_t) { return cudaErrorNoDevice; }
cudaError_t launch_scatter(const Geo &, const uint8_t *, const int32_t *, uint32_t, uint16_t *, cudaStream_t)
{ return cudaErrorNoDevice; }
cudaError_t launch_mirror_copy(const Geo &, const Work &, const uint16_t *, void *, uint32_t, int, uint32_t *, uint32_t,
                               cudaStream_t)
{ return cudaErrorNoDevice; }
cudaError_t launch_gather(const Geo &, const uint16_t *, const int32_t *, uint32_t, uint8_t *, cudaStream_t)
{ return cudaErrorNoDevice; }
cudaError_t launch_set(const void *, size_t, void *, cudaStream_t) { return cudaErrorNoDevice; }
cudaError_t launch_patch(const Geo &, int32_t *, kvs_record *, uint8_t *, const Patch *, uint32_t, cudaStream_t)
{ return cudaErrorNoDevice; }
cudaError_t launch_kivi_compress(const Geo &, const KiviJob *, uint32_t, const uint8_t *, uint8_t *, int32_t *,
                                 cudaStream_t) { return cudaErrorNoDevice; }
cudaError_t launch_decode_kivi(const Geo &, const Work &, const uint16_t *, const int32_t *, const uint8_t *,
                               uint32_t, int, cudaStream_t) { return cudaErrorNoDevice; }
int decode_kivi_blocks_per_sm(const Geo &) { return 0; }
cudaError_t launch_prefetch_plan(const PrefCand *, uint32_t, uint32_t, uint64_t *, uint64_t *, uint32_t *,
                                 cudaStream_t) { return cudaErrorNoDevice; }
cudaError_t launch_copy_mass(const Geo &, const Work &, const float *, float *, uint32_t, cudaStream_t)
{ return cudaErrorNoDevice; }
int decode_blocks_per_sm(const Geo &, uint32_t) { return 0; }
size_t decode_smem_bytes(const Geo &, uint32_t) { return 0; }

}  // namespace kvs
