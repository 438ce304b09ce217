"""dpclip on GB300: the per-linear-layer DP-SGD clipping path (exact, Hutch
and Hutch++ per-sample gradient norms, clip scales, clipped noisy gradient)
as hand-written sm_103a kernels behind a C ABI (include/dpclip.h).

`workloads` (seeded synthetic inputs) imports without the native library;
`api` and `_lib` need libdpclip.so and raise if it is missing.
"""
__version__ = "0.1.0"


def __getattr__(name):
    # Load the native library lazily so that `workloads` stays importable on a
    # host where the library has not been built yet.
    if name in ("api", "_lib"):
        import importlib
        return importlib.import_module(f".{name}", __name__)
    raise AttributeError(name)
