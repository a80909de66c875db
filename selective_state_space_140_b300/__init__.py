"""B300-native Mamba selective scan.

The compute path is the C-ABI library ``libmamba_scan.so`` (hand-written CUDA
for sm_103a, declared in ``include/mamba_scan.h``).  ``selective_state_space_140_b300.abi``
is its thin Python binding: it only marshals device pointers, sizes and the
stream into the C entry points, and it raises if the library is missing.

``selective_state_space_140_b300.workloads`` draws the seeded synthetic inputs.
"""

__all__ = ["abi", "workloads"]


def __getattr__(name):
    # Load the binding lazily so that importing the input generators never
    # needs the compiled library.
    if name == "abi":
        import importlib

        return importlib.import_module(".abi", __name__)
    raise AttributeError(name)
