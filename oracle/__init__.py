"""CPU oracle (test infrastructure only; see ``layout_oracle``)."""

from . import layout_oracle  # noqa: F401
