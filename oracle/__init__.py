"""fp64 CPU oracle of the Dobb optimizer step.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this
package: only the tests, the package's smoke check and the benchmark's CPU
baseline leg use it.  It shares no code with the CUDA implementation.

Every function cites the passage of "Dobb: Shard-Local Preconditioning in
Block-Diagonal Eigenbases" (arXiv 2610.39412) that it follows; see the module
headers of `oracle.dobb` and `oracle.metrics` for what pins each function.
"""
from . import dobb, metrics  # noqa: F401
