// Geometries (pure host functions) and launchers of the stage-1 kernels and
// the fold, shared by the C-ABI layer and the kernels that build on one
// another. Kept apart from conv_internal.h so that adding a kernel leaves the
// shared types (and the sources the recorded DRAM traffic is keyed on) as
// they are.
#pragma once

#include "conv_internal.h"

namespace cig {

// Kernel geometries (pure host functions).
Geometry geometry_generic(const Shape& s, conv_dir dir);
Geometry geometry_wgrad1x1_ffma(const Shape& s);
Geometry geometry_wgrad1x1_tf32x3(const Shape& s);
Geometry geometry_fwd_tc(const Shape& s);
Geometry geometry_fwd_tc_cluster(const Shape& s);
Geometry geometry_dgrad_tc(const Shape& s);
Geometry geometry_fwd_depthwise(const Shape& s);
Geometry geometry_fwd_grouped_tc(const Shape& s);
Geometry geometry_wgrad_grouped_tc(const Shape& s);
Geometry geometry_wgrad_tc(const Shape& s);
Geometry geometry_wgrad_grouped_mma(const Shape& s);
Geometry geometry_wgrad_depthwise_mma(const Shape& s);
Geometry geometry_fwd_grouped_mma(const Shape& s);
Geometry geometry_dgrad_grouped_mma(const Shape& s);
Geometry geometry_ffma(const Shape& s, conv_dir dir);
// The forward tensor-core kernel on a channel-block problem: output tile of
// channels [k0, k0 + 128) reads input channels [k0, k0 + 128) of X (full C
// for addressing) against a [K][R][S][128] filter; s.cg is 128 and s.groups 1.
Geometry geometry_fwd_tc_block(const Shape& block);
cudaError_t launch_fwd_tc_block(const Plan& p, const Args& a);
// The forward problem a stride-1, ungrouped data gradient equals (dY as the
// input, the transformed filter, padding dil * (f - 1) - pad).
Shape dgrad_as_forward(const Shape& s);
// The forward problem a stride-1 data gradient equals with its groups kept
// (dY as the input, C and K swapped, padding dil * (f - 1) - pad).
Shape dgrad_as_forward_grouped(const Shape& s);
Geometry geometry_dgrad_depthwise(const Shape& s);
Geometry geometry_dgrad_grouped_tc(const Shape& s);
Geometry geometry_wgrad_depthwise(const Shape& s);
Geometry geometry_wgrad_grouped(const Shape& s);

// Launchers: enqueue stage 1 on a.stream. Return the launch status.
cudaError_t launch_generic(const Plan& p, const Args& a);
cudaError_t launch_wgrad1x1_ffma(const Plan& p, const Args& a);
cudaError_t launch_wgrad1x1_tf32x3(const Plan& p, const Args& a);
cudaError_t launch_fwd_tc(const Plan& p, const Args& a);
cudaError_t launch_fwd_tc_cluster(const Plan& p, const Args& a);
cudaError_t launch_dgrad_tc(const Plan& p, const Args& a);
cudaError_t launch_fwd_depthwise(const Plan& p, const Args& a);
cudaError_t launch_fwd_grouped_tc(const Plan& p, const Args& a);
cudaError_t launch_wgrad_grouped_tc(const Plan& p, const Args& a);
cudaError_t launch_wgrad_tc(const Plan& p, const Args& a);
cudaError_t launch_wgrad_grouped_mma(const Plan& p, const Args& a);
cudaError_t launch_wgrad_depthwise_mma(const Plan& p, const Args& a);
cudaError_t launch_fwd_grouped_mma(const Plan& p, const Args& a);
cudaError_t launch_dgrad_grouped_mma(const Plan& p, const Args& a);
cudaError_t launch_ffma(const Plan& p, const Args& a);
cudaError_t launch_dgrad_depthwise(const Plan& p, const Args& a);
cudaError_t launch_dgrad_grouped_tc(const Plan& p, const Args& a);
cudaError_t launch_wgrad_depthwise(const Plan& p, const Args& a);
cudaError_t launch_wgrad_grouped(const Plan& p, const Args& a);
// Stage 2: out = cast(sum of slabs) (and the bias slabs into db).
cudaError_t launch_fold(const Plan& p, const Args& a);

}  // namespace cig
