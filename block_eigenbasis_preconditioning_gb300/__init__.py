"""Dobb optimizer step on one GB300 GPU (sm_103a CUDA kernels behind a C ABI).

"Dobb: Shard-Local Preconditioning in Block-Diagonal Eigenbases"
(arXiv 2610.39412).  `Dobb` is the optimizer object; `binding` exposes the
raw C ABI; `inputs` holds the seeded synthetic input generators.
"""
from .binding import DobbError, load_library, library_path  # noqa: F401


def __getattr__(name):
    # the optimizer needs torch; import it lazily so the generators and the
    # binding load without it
    if name == "Dobb":
        from .optimizer import Dobb
        return Dobb
    raise AttributeError(name)
