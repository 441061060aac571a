"""In-batch contrastive scoring on one GB300: the fused SigLIP sigmoid pair loss and hard MaxSim.

The compute path is the CUDA library built from `csrc/` (C ABI in `include/cli.h`);
`_binding` only marshals arguments to it and raises if the library is missing.
`synth` draws the seeded inputs.  The binding's names are re-exported lazily,
so `synth` imports without a built library.
"""

_BINDING_NAMES = {
    "CliError", "DeviceError", "InternalError", "InvalidArgumentError", "MalformedError", "ShapeMismatchError",
    "UnsupportedError", "check_device_status", "device_edges", "maxsim_backward", "maxsim_backward_workspace_bytes",
    "maxsim_scores", "maxsim_workspace_bytes", "pair_loss_sigmoid_fwd_bwd", "pair_loss_sigmoid_scores_fwd_bwd",
    "pair_loss_sigmoid_scores_workspace_bytes", "pair_loss_sigmoid_workspace_bytes", "status_name", "LIB_PATH",
    "raise_for", "pair_loss_scores_fwd_bwd", "pair_loss_scores_workspace_bytes",
    "pair_loss_sigmoid_matryoshka_fwd_bwd", "pair_loss_sigmoid_matryoshka_workspace_bytes",
    "pair_loss_sigmoid_groups_fwd_bwd", "maxsim_scores_named", "maxsim_named_workspace_bytes",
    "maxsim_backward_named", "selftest_bounded_wait",
}


def __getattr__(name):
    if name in _BINDING_NAMES:
        from . import _binding
        return getattr(_binding, name)
    raise AttributeError(name)
