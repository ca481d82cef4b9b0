"""fp64 CPU oracle of the InfLLM v2 path -- test infrastructure only.

Imported by the tests, by the package's smoke check and by the benchmark's
CPU-baseline leg; never by the product path.  See ``infllmv2_oracle``.
"""

from .infllmv2_oracle import *  # noqa: F401,F403
from .infllmv2_oracle import Settings, Selection  # noqa: F401
